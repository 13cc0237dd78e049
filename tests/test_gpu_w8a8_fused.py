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
from _helpers import bf16_to_f64, check_tol, from_dev_bf16, to_dev, to_dev_bf16

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


# ---------------------------------------------------------------- FP8 (E4M3)
# From 64 token tiles (M > 8064), K >= 4096, for GEMMs of at most 4096 columns
# whose tile pairs fill the SMs, the E4M3 W8A8 linear is one kernel too: warps of every
# GEMM CTA quantize the activations into the codes workspace, task by task, and
# the TMA producer waits on each task's flag (or its band's count) before
# loading those codes, so the quantization overlaps the tensor-core work.

def _run_e4m3(capi, M, K, N, tag, x_scale_mult=1.0, with_bias=False, glu=False):
    rng = synth.rng_for("test-w8a8-fused", 0, f"e4m3-{M}x{K}x{N}-{tag}", "all")
    outl = synth.outlier_channels(K, rng)
    rows_w = 2 * N if glu else N
    w = synth.weights(rows_w, K, rng)
    cal = synth.activations(512, K, rng, outl)
    x = synth.activations(M, K, rng, outl)
    if x_scale_mult != 1.0:
        x = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x) * np.float32(x_scale_mult))
    b = synth.bias(rows_w, rng) if with_bias else None
    q, s = oracle.quantize_weight(oracle.E4M3, w)
    sx = oracle.act_scale(oracle.E4M3, cal)
    op = capi.QLIN_OP_W8A8_GATE_UP_SILU if glu else capi.QLIN_OP_W8A8_LINEAR
    assert capi.qlin_kernel_name(op, "e4m3", M, K, N) == "k_fp8_gemm<xq>"
    fn = capi.w8a8_gate_up_silu if glu else capi.w8a8_linear
    y = fn("e4m3", to_dev_bf16(x), to_dev(np.array([sx], np.float32)), to_dev(q), to_dev(s),
           None if b is None else to_dev_bf16(b))
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 24)), [M - 1]]))
    qx = oracle.quantize_act(oracle.E4M3, x, sx)
    ref = (oracle.w8a8_gate_up_silu if glu else oracle.w8a8)(oracle.E4M3, qx, sx, q, s, b, rows=rows)
    check_tol(from_dev_bf16(y)[rows], ref, f"fused e4m3 {M}x{K}x{N} {tag}")


@pytest.mark.parametrize("M,K,N", [(8192, 4096, 2048), (8193, 4112, 2304), (8200, 4224, 1024),
                                   (8192, 11008, 2048)])
def test_fused_e4m3_w8a8_shapes(capi, M, K, N):
    _run_e4m3(capi, M, K, N, "shapes", with_bias=(K % 128 != 0))


def test_fused_e4m3_w8a8_beyond_calibration_range(capi):
    _run_e4m3(capi, 8320, 4096, 4096, "clamp", x_scale_mult=40.0)


def test_fused_e4m3_gate_up_silu(capi):
    _run_e4m3(capi, 8192, 4096, 1024, "glu", glu=True, with_bias=True)


@pytest.mark.parametrize("M,K,N", [(8193, 4112, 2048), (8320, 4096, 4096)])
def test_fused_e4m3_codes_bitexact(capi, M, K, N):
    """The in-GEMM quantizer leaves its codes in the workspace's first M*K bytes:
    they must equal the oracle's static E4M3 quantization bit for bit, here with
    signed zeros and values far beyond the calibration range mixed in."""
    rng = synth.rng_for("test-w8a8-fused", 0, f"e4m3-codes-{M}x{K}", "all")
    x = synth.activations(M, K, rng, synth.outlier_channels(K, rng))
    xf = synth.bf16_bits_to_f32(x)
    pick = rng.random(xf.shape)
    xf = np.where(pick < 0.01, np.float32(-0.0), xf)
    xf = np.where((pick > 0.99) & (pick < 0.995), xf * np.float32(3e4), xf)
    x = synth.f32_to_bf16_bits(xf)
    w = synth.weights(N, K, rng)
    q, s = oracle.quantize_weight(oracle.E4M3, w)
    sx = oracle.act_scale(oracle.E4M3, synth.activations(512, K, rng))
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, "e4m3", M, K, N) == "k_fp8_gemm<xq>"
    xd = to_dev_bf16(x)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = capi.workspace(capi.QLIN_OP_W8A8_LINEAR, "e4m3", M, K, N, device=xd.device)
    capi.qlin_w8a8_linear("e4m3", xd, to_dev(np.array([sx], np.float32)), to_dev(q), to_dev(s), None, y, ws)
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    got = ws.view(torch.uint8)[: M * K].cpu().numpy().reshape(M, K)
    ref = oracle.quantize_act(oracle.E4M3, x, sx)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:4].tolist()}"
    assert (ref == 0x80).any() and (ref == 0xFE).any()  # -0 and -448 both occur


@pytest.mark.parametrize("M", [1, 16, 33, 64])
def test_fused_int8_codes_bitexact(capi, M):
    """The codes the fused kernel quantizes in place, read back bit for bit: an
    identity weight (code 1 on the diagonal, scale 1, no bias) makes every output
    y[m, n] = code[m, n] * s_x, and with s_x = 2^-4 that product is exact in BF16.
    The activations include exact ties (half-integers times s_x, which round to
    even), values beyond the clamp (N(0, 9) spans +-48 s_x per sigma, and +-300),
    zeros and negative zeros; the codes must equal the oracle's."""
    K = N = 512
    sx = np.float32(2.0 ** -4)
    rng = synth.rng_for("test-w8a8-fused", 0, f"codes-{M}", "all")
    xf = (rng.standard_normal((M, K)) * 3.0).astype(np.float32)
    halves = (rng.integers(-127, 127, size=(M, K)) + 0.5).astype(np.float32) * sx  # exact ties in BF16
    pick = rng.random((M, K)) < 0.3
    xf = np.where(pick, halves, xf)
    xf[:, :4] = np.array([0.0, -0.0, 300.0, -300.0], np.float32)
    x = synth.f32_to_bf16_bits(xf)
    qw = np.eye(N, K, dtype=np.int8).view(np.uint8)
    sw = np.ones(N, np.float32)
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, "int8", M, K, N).endswith(",i8,xq>")
    y = capi.w8a8_linear("int8", to_dev_bf16(x), to_dev(np.array([sx], np.float32)), to_dev(qw), to_dev(sw), None)
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    codes = bf16_to_f64(from_dev_bf16(y)) / float(sx)
    assert np.all(codes == np.round(codes))
    ref = oracle.quantize_act(oracle.INT8, x, sx).view(np.int8).astype(np.float64)
    bad = np.argwhere(codes != ref)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:4].tolist()}"
    assert (np.abs(ref) == 127).any() and (ref == 0).any()
