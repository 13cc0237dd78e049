"""INT8 W8A8 static linear with the activation quantization fused into the GEMM (GPU).

For one token tile (M <= 64) qlin_w8a8_linear runs a single kernel: the
converter warps quantize each BF16 activation tile in place with the static
scale before the tensor cores read it.  These tests hold it to the oracle
(quantize with the same scale, exact int32 accumulator, fp64 epilogue) at the
tile-size edges, with activations far beyond the calibration range (clamped
codes), with a tiny scale (the exact-division path of the quotient), with
bias, for the merged gate_up form, and check the launch is the fused kernel.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_quantized_linear_gb300 import synth
from _helpers import check_tol, from_dev_bf16, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    from bit_quantized_linear_gb300 import capi as c
    return c


def _run(capi, M, K, N, tag, x_scale_mult=1.0, sx_override=None, with_bias=True):
    rng = synth.rng_for("test-w8a8-fused", 0, f"{M}x{K}x{N}-{tag}", "all")
    outl = synth.outlier_channels(K, rng)
    w = synth.weights(N, K, rng)
    cal = synth.activations(512, K, rng, outl)
    x = synth.activations(M, K, rng, outl)
    if x_scale_mult != 1.0:
        x = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x) * np.float32(x_scale_mult))
    b = synth.bias(N, rng) if with_bias else None
    q, s = oracle.quantize_weight(oracle.INT8, w)
    sx = oracle.act_scale(oracle.INT8, cal) if sx_override is None else np.float32(sx_override)
    y = capi.w8a8_linear("int8", to_dev_bf16(x), to_dev(np.array([sx], np.float32)), to_dev(q), to_dev(s),
                         None if b is None else to_dev_bf16(b))
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    qx = oracle.quantize_act(oracle.INT8, x, sx)
    ref = oracle.w8a8(oracle.INT8, qx, sx, q, s, b)
    check_tol(from_dev_bf16(y), ref, f"fused w8a8 {M}x{K}x{N} {tag}")
    return qx


@pytest.mark.parametrize("M", [1, 15, 16, 17, 32, 33, 63, 64])
def test_fused_int8_w8a8_tile_edges(capi, M):
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, "int8", M, 2048, 512).endswith(",i8,xq>")
    _run(capi, M, 2048, 512, "edges")


def test_fused_int8_w8a8_beyond_calibration_range(capi):
    """Run-time activations 40x the calibration batch: many codes clamp at +-127."""
    qx = _run(capi, 16, 1024, 384, "clamp", x_scale_mult=40.0)
    assert (np.abs(qx.view(np.int8)) == 127).mean() > 0.02


def test_fused_int8_w8a8_tiny_scale_takes_exact_division(capi):
    """A scale below 2^-96 takes the IEEE division inside the quotient; with it every
    nonzero code saturates."""
    qx = _run(capi, 8, 512, 256, "tiny", sx_override=2.0 ** -100, with_bias=False)
    assert (np.abs(qx.view(np.int8)) == 127).mean() > 0.9


@pytest.mark.parametrize("M,K,N", [(1, 11008, 2048), (16, 2048, 11008), (64, 3584, 3584)])
def test_fused_int8_w8a8_3b_7b_shapes(capi, M, K, N):
    _run(capi, M, K, N, "shapes", with_bias=(M == 16))


def test_fused_int8_gate_up_silu(capi):
    M, K, I = 24, 1024, 256
    rng = synth.rng_for("test-w8a8-fused", 0, "glu", "all")
    w = synth.weights(2 * I, K, rng)
    cal = synth.activations(512, K, rng)
    x = synth.activations(M, K, rng)
    q, s = oracle.quantize_weight(oracle.INT8, w)
    sx = oracle.act_scale(oracle.INT8, cal)
    y = capi.w8a8_gate_up_silu("int8", to_dev_bf16(x), to_dev(np.array([sx], np.float32)), to_dev(q), to_dev(s))
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    ref = oracle.w8a8_gate_up_silu(oracle.INT8, oracle.quantize_act(oracle.INT8, x, sx), sx, q, s)
    check_tol(from_dev_bf16(y), ref, "fused int8 gate_up silu")
