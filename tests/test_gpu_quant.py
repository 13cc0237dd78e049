"""GPU parity of the quantizers against the oracle: bit-exact codes and scales."""
import numpy as np
import pytest
import torch

import oracle
from bit_quantized_linear_gb300 import synth
from _helpers import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
QT = {"int8": oracle.INT8, "e4m3": oracle.E4M3}


@pytest.fixture(scope="module")
def capi():
    from bit_quantized_linear_gb300 import capi as c
    return c


def _gpu_quant_weight(capi, qt, w):
    qw, s = capi.quantize_weight(qt, to_dev(w))
    torch.cuda.synchronize()
    return qw.cpu().numpy(), s.cpu().numpy()


def _assert_weight_parity(capi, qt, w):
    q, s = _gpu_quant_weight(capi, qt, w)
    oq, os_ = oracle.quantize_weight(QT[qt], w)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32)), "scale bits differ"
    diff = np.nonzero(q != oq)
    assert diff[0].size == 0, f"{diff[0].size} codes differ, first at {diff[0][0], diff[1][0]}: " \
                              f"gpu {q[diff][0]:#x} oracle {oq[diff][0]:#x} w={w[diff][0]!r}"


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("N,K", [(16, 16), (48, 80), (1024, 1024), (257, 3584), (64, 18944)])
def test_quantize_weight_bitexact(capi, qt, N, K):
    rng = synth.rng_for("test-qw", 0, f"{N}x{K}", qt)
    _assert_weight_parity(capi, qt, synth.weights(N, K, rng))


@pytest.mark.parametrize("name,K,N", [("q_proj", 3584, 3584), ("gate_up_proj", 3584, 37888),
                                      ("down_proj", 18944, 3584)])
def test_quantize_weight_decode7b_full(capi, name, K, N):
    lin = synth.Linear(name, K, N, 1, "e4m3", "w8a16", outliers=True, workload=synth.DECODE7B)
    w = synth.make_inputs(lin, want=("w",))["w"]
    _assert_weight_parity(capi, "e4m3", w)


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_quantize_weight_special_rows(capi, qt):
    K = 64
    w = np.zeros((6, K), np.float32)
    w[1] = np.eye(K, dtype=np.float32)[3]                     # one-hot
    w[2] = np.linspace(-5, 5, K, dtype=np.float32)            # many exact midpoints
    w[3, :4] = [127, 2.5, -0.5, 1.5]                          # ties to even (s = 1 for INT8)
    w[4] = np.float32(1e-30) * np.arange(K, dtype=np.float32)  # tiny magnitudes
    w[5] = -np.float32(3e4)
    _assert_weight_parity(capi, qt, w)


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_quantize_weight_midpoints(capi, qt):
    """Rows whose elements sit on and next to every rounding midpoint of the
    target grid (times the row scale): exercises ties-to-even and the division."""
    e4 = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    mids = (np.arange(-126, 127) + 0.5) if qt == "int8" else np.concatenate(
        [(e4[:-1] + e4[1:]) / 2, -(e4[:-1] + e4[1:]) / 2])
    qmax = 127.0 if qt == "int8" else 448.0
    rng = np.random.default_rng(5)
    rows = []
    for _ in range(32):
        amax = np.float32(rng.uniform(0.01, 4.0))
        s = amax / np.float32(qmax)
        base = (mids * np.float64(s)).astype(np.float32)
        r = np.concatenate([[amax], base, np.nextafter(base, np.float32(9e9)), np.nextafter(base, np.float32(-9e9))])
        r = np.clip(r, -amax, amax).astype(np.float32)
        pad = (-len(r)) % 16
        rows.append(np.concatenate([r, np.zeros(pad, np.float32)]))
    _assert_weight_parity(capi, qt, np.stack(rows))


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("rows,K", [(1, 16), (7, 48), (512, 2048), (synth.CALIB_ROWS, 2048)])
def test_act_scale_bitexact(capi, qt, rows, K):
    rng = synth.rng_for("test-cal", 0, f"{rows}x{K}", qt)
    outl = synth.outlier_channels(K, rng)
    x = synth.activations(rows, K, rng, outl)
    s = capi.act_scale_from_calib(qt, to_dev_bf16(x)).cpu().numpy()[0]
    assert np.float32(s).view(np.uint32) == oracle.act_scale(QT[qt], x).view(np.uint32)


def test_act_scale_zero_batch(capi):
    for qt in ("int8", "e4m3"):
        s = capi.act_scale_from_calib(qt, torch.zeros((4, 32), dtype=torch.bfloat16, device="cuda"))
        assert s.item() == 1.0


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M,K", [(1, 16), (3, 2048), (16, 11008), (1024, 2048)])
def test_quantize_act_bitexact(capi, qt, M, K):
    rng = synth.rng_for("test-qa", 0, f"{M}x{K}", qt)
    outl = synth.outlier_channels(K, rng)
    cal = synth.activations(256, K, rng, outl)
    x = synth.activations(M, K, rng, outl)
    s = oracle.act_scale(QT[qt], cal)
    qx = capi.quantize_act_static(qt, to_dev_bf16(x), to_dev(np.array([s], np.float32))).cpu().numpy()
    oq = oracle.quantize_act(QT[qt], x, s)
    assert np.array_equal(qx, oq), f"{int((qx != oq).sum())} codes differ"


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_quantize_act_clamps_beyond_calibration(capi, qt):
    """Run-time activations larger than the calibration maximum clamp/saturate."""
    x = synth.f32_to_bf16_bits(np.array([[1.0, -3.0, 300.0, -1e4, 0.5, 1.5, -0.0, 2.5] * 2], np.float32))
    for s in (np.float32(1.0), np.float32(0.5), np.float32(0.0123)):
        qx = capi.quantize_act_static(qt, to_dev_bf16(x), to_dev(np.array([s], np.float32))).cpu().numpy()
        assert np.array_equal(qx, oracle.quantize_act(QT[qt], x, s))


def test_e4m3_all_bf16_values(capi):
    """Every finite BF16 value (x 1/1 scale) through the E4M3 activation cast,
    and through the INT8 one: covers every binade, subnormals and saturation."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_bits_to_f32(bits)
    bits = bits[np.isfinite(f)]
    bits = np.concatenate([bits, np.zeros((-len(bits)) % 16, np.uint16)]).reshape(-1, 16)
    for qt, s in (("e4m3", np.float32(1.0)), ("e4m3", np.float32(0.37)), ("int8", np.float32(1.0)),
                  ("int8", np.float32(2.0 ** -100))):
        qx = capi.quantize_act_static(qt, to_dev_bf16(bits), to_dev(np.array([s], np.float32))).cpu().numpy()
        assert np.array_equal(qx, oracle.quantize_act(QT[qt], bits, s)), (qt, s)
