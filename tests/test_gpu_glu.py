"""Merged gate_up linear with the fused SiLU * up epilogue against the oracle (GPU).

y[m, n] = silu(g) * u, g and u the linear's outputs for gate row n and up row
I + n of the merged [2I, K] weight.  The oracle computes the fp64 result on the
same quantized operands; the BF16 output must meet the layer's tolerance.
Shapes cover every token-tile size of the decode kernel (16..256), the
split-K cluster path (few output tiles) and the single-CTA path, the FP8 and
INT8 W8A8 kernels, bias and no bias, and the full-size 7B and 3B-stack MLPs on
sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_quantized_linear_gb300 import synth
from _helpers import check_tol, from_dev_bf16, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
QT = {"int8": oracle.INT8, "e4m3": oracle.E4M3}


@pytest.fixture(scope="module")
def capi():
    from bit_quantized_linear_gb300 import capi as c
    return c


def _case(qt, M, K, I, with_bias, tag, cal_rows=0):
    rng = synth.rng_for("test-glu", 0, f"{qt}-{M}x{K}x{I}-{tag}", "all")
    outl = synth.outlier_channels(K, rng)
    w = synth.weights(2 * I, K, rng)
    x = synth.activations(M, K, rng, outl)
    b = synth.bias(2 * I, rng) if with_bias else None
    cal = synth.activations(cal_rows, K, rng, outl) if cal_rows else None
    q, s = oracle.quantize_weight(QT[qt], w)
    return x, q, s, b, cal


def _status_ok(capi):
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK


def w8a16_glu(capi, qt, M, K, I, with_bias, tag, rows=None):
    x, q, s, b, _ = _case(qt, M, K, I, with_bias, tag)
    y = capi.w8a16_gate_up_silu(qt, to_dev_bf16(x), to_dev(q), to_dev(s), None if b is None else to_dev_bf16(b))
    _status_ok(capi)
    y = from_dev_bf16(y)
    ref = oracle.w8a16_gate_up_silu(QT[qt], x, q, s, b, rows=rows)
    check_tol(y if rows is None else y[rows], ref, f"w8a16 glu {qt} {M}x{K}x{I}")


def w8a8_glu(capi, qt, M, K, I, with_bias, tag, rows=None):
    x, q, s, b, cal = _case(qt, M, K, I, with_bias, tag, cal_rows=512)
    sx = oracle.act_scale(QT[qt], cal)
    y = capi.w8a8_gate_up_silu(qt, to_dev_bf16(x), to_dev(np.array([sx], np.float32)), to_dev(q), to_dev(s),
                               None if b is None else to_dev_bf16(b))
    _status_ok(capi)
    y = from_dev_bf16(y)
    qx = oracle.quantize_act(QT[qt], x, sx)
    ref = oracle.w8a8_gate_up_silu(QT[qt], qx, sx, q, s, b, rows=rows)
    check_tol(y if rows is None else y[rows], ref, f"w8a8 glu {qt} {M}x{K}x{I}")


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M,K,I", [(1, 512, 128), (16, 1024, 256), (33, 3584, 384), (64, 640, 128),
                                   (128, 2048, 640), (200, 1024, 128), (256, 512, 4096), (300, 512, 256)])
def test_w8a16_gate_up_silu(capi, qt, M, K, I):
    w8a16_glu(capi, qt, M, K, I, M % 2 == 0, "a")


@pytest.mark.parametrize("M,K,I", [(1, 1040, 384), (3, 3584, 256), (6, 18944, 128), (8, 3584, 256),
                                   (16, 3584, 128), (29, 528, 2048), (32, 2048, 640)])
def test_w8a16_gate_up_silu_e4m3_fp8_path(capi, M, K, I):
    """E4M3 up to 32 tokens: a weight tile is 64 gate rows and their 64 up rows,
    so gate and up meet in one partial tile before silu(g) * u is formed."""
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A16_GATE_UP_SILU, "e4m3", M, K, I).startswith("k_w8a16_split+")
    w8a16_glu(capi, "e4m3", M, K, I, M % 2 == 0, "f8")


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M,K,I", [(1, 256, 128), (40, 1024, 256), (64, 512, 8192), (130, 2048, 384),
                                   (1000, 1024, 512)])
def test_w8a8_gate_up_silu(capi, qt, M, K, I):
    w8a8_glu(capi, qt, M, K, I, M % 2 == 1, "b")


@pytest.mark.parametrize("qt,M", [("e4m3", 1), ("e4m3", 256), ("int8", 32)])
def test_w8a16_gate_up_silu_7b_full(capi, qt, M):
    """Qwen2.5-7B MLP: hidden 3584, intermediate 18944 (merged weight 37888 x 3584)."""
    w8a16_glu(capi, qt, M, 3584, 18944, False, "7b", rows=sample_rows(M, 8))


def test_w8a8_gate_up_silu_stack_prefill(capi):
    """The 3B stack's prefill MLP: M = 8192, hidden 2048, intermediate 11008, E4M3."""
    w8a8_glu(capi, "e4m3", 8192, 2048, 11008, False, "stack", rows=sample_rows(8192, 12))


def test_gate_up_silu_zero_tokens(capi):
    I, K = 128, 64
    q = torch.zeros((2 * I, K), dtype=torch.uint8, device="cuda")
    s = torch.ones(2 * I, device="cuda")
    x = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    n0 = capi.qlin_launch_count()
    y = capi.w8a16_gate_up_silu("int8", x, q, s)
    assert y.shape == (0, I) and capi.qlin_launch_count() == n0


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_w8a16_gate_up_silu_partial_last_wave(capi, qt):
    """Merged gate_up with a mostly empty last wave of units (I = 11008 at 256
    tokens: 344 units of 64 gate + 64 up rows on 152 persistent CTAs).  Full
    output against the oracle."""
    w8a16_glu(capi, qt, 256, 2048, 11008, True, "last-wave")
