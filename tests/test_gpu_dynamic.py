"""GPU parity of the dynamic per-token W8A8 path against the oracle: codes and
per-token scales bit-exact, BF16 outputs within the stated tolerance."""
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


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M,K", [(1, 16), (5, 48), (129, 2048), (1024, 11008)])
def test_quantize_act_dynamic_bitexact(capi, qt, M, K):
    rng = synth.rng_for("test-dyn", 0, f"{M}x{K}", qt)
    xf = synth.bf16_bits_to_f32(synth.activations(M, K, rng, synth.outlier_channels(K, rng)))
    xf[M // 2] = 0.0  # an all-zero token row
    x = synth.f32_to_bf16_bits(xf)
    qx, s = capi.quantize_act_dynamic(qt, to_dev_bf16(x))
    oq, os_ = oracle.quantize_act_per_token(QT[qt], x)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(qx.cpu().numpy(), oq)


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M,K,N", [(1, 16, 16), (3, 2048, 2048), (16, 2048, 11008), (130, 1040, 400),
                                   (256, 11008, 2048), (1024, 2048, 11008)])
def test_w8a8_dynamic_linear(capi, qt, M, K, N):
    rng = synth.rng_for("test-dyn-lin", 0, f"{qt}-{M}x{K}x{N}", "all")
    x = synth.activations(M, K, rng, synth.outlier_channels(K, rng))
    q, s = oracle.quantize_weight(QT[qt], synth.weights(N, K, rng))
    b = synth.bias(N, rng)
    y = capi.w8a8_dynamic_linear(qt, to_dev_bf16(x), to_dev(q), to_dev(s), to_dev_bf16(b))
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    rows = None if M <= 130 else sample_rows(M, 24)
    qx, sx = oracle.quantize_act_per_token(QT[qt], x)
    ref = oracle.w8a8_per_token(QT[qt], qx, sx, q, s, b, rows=rows)
    yb = from_dev_bf16(y)
    check_tol(yb if rows is None else yb[rows], ref, f"dynamic {qt} {M}x{K}x{N}")


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_w8a8_dynamic_row_scaling(capi, qt):
    """Scaling one token row by 2^j scales only that output row, bit-exactly."""
    rng = np.random.default_rng(71)
    M, K, N = 40, 512, 256
    xf = synth.bf16_bits_to_f32(synth.activations(M, K, rng))
    q, s = oracle.quantize_weight(QT[qt], synth.weights(N, K, rng))
    y1 = synth.bf16_bits_to_f32(from_dev_bf16(capi.w8a8_dynamic_linear(
        qt, to_dev_bf16(synth.f32_to_bf16_bits(xf)), to_dev(q), to_dev(s))))
    xf[7] *= np.float32(4)
    y2 = synth.bf16_bits_to_f32(from_dev_bf16(capi.w8a8_dynamic_linear(
        qt, to_dev_bf16(synth.f32_to_bf16_bits(xf)), to_dev(q), to_dev(s))))
    assert np.array_equal(y2[7], 4 * y1[7])
    assert np.array_equal(np.delete(y2, 7, 0), np.delete(y1, 7, 0))
