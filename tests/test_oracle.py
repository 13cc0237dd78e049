"""Pins for the CPU oracle (not gpu).

Each test checks the oracle against something other than its own code: hand
worked fixtures (tests/golden), brute-force search, closed forms, invariants,
exact rational arithmetic, or an independent library cast (torch's CPU
float8_e4m3fn conversion).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from bit_quantized_linear_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
INT8, E4M3 = 0, 1


def _num(t):
    t = t.strip()
    return int(t, 16) if t.lower().startswith("0x") else float(t)


# ---------------------------------------------------------------- E4M3 codec
def e4m3_points():
    codes, nans, rounds = [], [], []
    for line in open(os.path.join(GOLDEN, "e4m3_points.txt")):
        line = line.split("#")[0].split()
        if not line:
            continue
        if line[0] == "code":
            codes.append((int(line[1], 16), float(line[3])))
        elif line[0] == "nan":
            nans.append(int(line[1], 16))
        elif line[0] == "round":
            rounds.append((float(line[1]), int(line[3], 16)))
    return codes, nans, rounds


def test_e4m3_golden_points(orc):
    codes, nans, rounds = e4m3_points()
    for c, v in codes:
        d = orc.e4m3_decode(c)
        assert d == v and math.copysign(1, d) == math.copysign(1, v), (hex(c), d, v)
    for c in nans:
        assert math.isnan(orc.e4m3_decode(c))
    for v, c in rounds:
        assert orc.e4m3_encode(v) == c, (v, hex(orc.e4m3_encode(v)), hex(c))


def test_e4m3_decode_matches_torch_cast(orc):
    """All 256 codes against torch's CPU float8_e4m3fn -> float32 conversion."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        d = orc.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(d), hex(c)
        else:
            assert d == ref[c], (hex(c), d, ref[c])


def test_e4m3_roundtrip_and_monotone(orc):
    vals = []
    for c in range(256):
        d = orc.e4m3_decode(c)
        if math.isnan(d):
            continue
        assert orc.e4m3_encode(d) == c, hex(c)  # +0 and -0 stay distinct
        if c < 0x80:
            vals.append(d)
    assert all(b > a for a, b in zip(vals, vals[1:]))  # positive codes strictly increase
    assert len(vals) == 127


def test_e4m3_midpoints_round_to_even(orc):
    pos = [orc.e4m3_decode(c) for c in range(0x7F)]
    for c in range(0x7E):
        mid = (pos[c] + pos[c + 1]) / 2
        want = c if c % 2 == 0 else c + 1
        assert orc.e4m3_encode(mid) == want, (hex(c), mid)
        assert orc.e4m3_encode(-mid) == 0x80 | want
        # just off the midpoint goes to the nearer neighbour
        assert orc.e4m3_encode(np.nextafter(mid, 0)) == c
        assert orc.e4m3_encode(np.nextafter(mid, 1e9)) == c + 1


def test_e4m3_encode_matches_torch_cast_in_range(orc):
    """Random fp32 values across all binades, |v| < 464 (where torch does not
    produce NaN): the oracle's encoder equals torch's round-to-nearest-even cast."""
    rng = np.random.default_rng(123)
    mag = np.exp2(rng.uniform(-12, math.log2(463.9), 20000)).astype(np.float32)
    sgn = np.where(rng.random(20000) < 0.5, -1, 1).astype(np.float32)
    v = mag * sgn
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(a)) for a in v], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_saturation(orc):
    for v in [448.0, 449.0, 464.0, 480.0, 1e6, 3.0e38]:
        assert orc.e4m3_encode(v) == 0x7E
        assert orc.e4m3_encode(-v) == 0xFE


# ------------------------------------------------------------ INT8 quantizer
def int8_rows():
    out = []
    for line in open(os.path.join(GOLDEN, "int8_rounding.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        parts = [p.split() for p in line.split("|")]
        row = np.array([float(t) for t in parts[0][1:]], np.float32)
        scale = np.float32(float(parts[1][1]))
        q = np.array([int(t) for t in parts[2][1:]], np.int8)
        out.append((row, scale, q))
    return out


def test_int8_golden_rows(orc):
    for row, scale, q in int8_rows():
        got_q, got_s = orc.quantize_weight(INT8, row[None, :])
        assert got_s[0] == scale, (row, got_s[0], scale)
        assert np.array_equal(got_q[0].view(np.int8), q), (row, got_q[0].view(np.int8), q)


def _brute_int(v):
    """Nearest integer in [-127,127] to v by exhaustive search; ties to even."""
    cands = np.arange(-127, 128)
    d = np.abs(cands.astype(np.float64) - float(v))
    best = d.min()
    tie = cands[d == best]
    return int(tie[tie % 2 == 0][0]) if len(tie) > 1 else int(tie[0])


def test_int8_bruteforce_small(orc):
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((6, 40)) * rng.uniform(0.01, 10, (6, 1))).astype(np.float32)
    w[2, 5] = np.float32(-3.5) * np.abs(w[2]).max() / 127  # exercise sign / ties a bit
    q, s = orc.quantize_weight(INT8, w)
    for n in range(w.shape[0]):
        assert s[n] == np.float32(np.abs(w[n]).max()) / np.float32(127)
        for k in range(w.shape[1]):
            v = np.float32(w[n, k]) / s[n]
            assert q[n, k].view(np.int8) == _brute_int(v)


def test_int8_roundtrip_bound_and_extremes(orc):
    rng = np.random.default_rng(11)
    N, K = 64, 3584
    w = synth.weights(N, K, rng)
    q, s = orc.quantize_weight(INT8, w)
    qi = q.view(np.int8).astype(np.float64)
    sd = s.astype(np.float64)[:, None]
    err = np.abs(w.astype(np.float64) - sd * qi)
    assert np.all(err <= sd / 2 + sd * 2.0 ** -17)
    assert np.abs(qi).max() <= 127
    # each row's largest-magnitude element maps to +-127 exactly
    idx = np.abs(w).argmax(axis=1)
    assert np.all(np.abs(qi[np.arange(N), idx]) == 127)


def test_int8_identity_and_zero_rows(orc):
    K = 48
    w = np.eye(K, dtype=np.float32)
    q, s = orc.quantize_weight(INT8, w)
    assert np.all(q.view(np.int8) == 127 * np.eye(K, dtype=np.int8))
    assert np.all(s == np.float32(1) / np.float32(127))
    z = np.zeros((3, 32), np.float32)
    q, s = orc.quantize_weight(INT8, z)
    assert np.all(s == 1.0) and np.all(q == 0)


def test_int8_reconstruction_band(orc):
    """Statistical sanity band: relative L2 reconstruction error of N(0,1/K)
    weights is about E[max|row|] * sqrt(K) / (127 * sqrt(12)); the tiny-vllm README
    ("Quality Check", artifact check) reports 0.00949 on real Qwen3-0.6B layers."""
    rng = np.random.default_rng(0)
    for K in (1024, 3584):
        w = synth.weights(256, K, rng)
        q, s = orc.quantize_weight(INT8, w)
        rec = s[:, None].astype(np.float64) * q.view(np.int8)
        rel = np.linalg.norm(w - rec) / np.linalg.norm(w)
        pred = np.abs(w).max(axis=1).mean() * math.sqrt(K) / (127 * math.sqrt(12))
        assert abs(rel - pred) / pred < 0.03
        assert 0.004 < rel < 0.015


# ------------------------------------------------------------ E4M3 quantizer
def _all_codes(orc):
    return [(c, orc.e4m3_decode(c)) for c in range(256) if not math.isnan(orc.e4m3_decode(c))]


def _brute_e4m3(v, table):
    """Exhaustive nearest code (ties to even mantissa), saturating beyond 448."""
    if v >= 448:
        return 0x7E
    if v <= -448:
        return 0xFE
    best = min(abs(d - v) for _, d in table)
    cands = [c for c, d in table if abs(d - v) == best]
    if v == 0:
        return 0x80 if math.copysign(1, v) < 0 else 0x00
    cands = [c for c in cands if (c & 0x80) == (0x80 if v < 0 else 0)]
    if len(cands) > 1:
        cands = [c for c in cands if c % 2 == 0]
    return cands[0]


def test_e4m3_weight_bruteforce_small(orc):
    table = _all_codes(orc)
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((5, 24)) * np.array([[1e-3], [0.1], [1], [30], [1e4]])).astype(np.float32)
    q, s = orc.quantize_weight(E4M3, w)
    for n in range(5):
        assert s[n] == np.float32(np.abs(w[n]).max()) / np.float32(448)
        for k in range(24):
            v = float(np.float32(w[n, k]) / s[n])
            assert q[n, k] == _brute_e4m3(v, table), (n, k, v)
        assert (q[n, np.abs(w[n]).argmax()] & 0x7F) == 0x7E


def test_e4m3_weight_exact_grid_rows(orc):
    """A row already on the E4M3 grid with max 448 quantizes to itself (s = 1)."""
    vals = np.array([448, 17, 19, 1.5 * 2 ** -9, 0, -240, 2 ** -6], np.float32)
    q, s = orc.quantize_weight(E4M3, vals[None, :])
    assert s[0] == 1.0
    assert list(q[0]) == [0x7E, 0x58, 0x5A, 0x02, 0x00, 0xF7, 0x08]


# ------------------------------------------------------- activations / calib
def test_act_scale_closed_forms(orc):
    x = np.zeros((4, 16), np.float32)
    x[2, 3] = -254.0
    xb = synth.f32_to_bf16_bits(x)
    assert orc.act_scale(INT8, xb) == np.float32(2.0)
    x[2, 3] = 896.0
    assert orc.act_scale(E4M3, synth.f32_to_bf16_bits(x)) == np.float32(2.0)
    assert orc.act_scale(INT8, np.zeros((2, 16), np.uint16)) == np.float32(1.0)


def test_act_quant_clamp_and_saturation(orc):
    x = synth.f32_to_bf16_bits(np.array([[1.0, -3.0, 300.0, -1e4, 0.5, 1.5, -0.0]], np.float32))
    q = orc.quantize_act(INT8, x, np.float32(1.0))
    assert list(q[0].view(np.int8)) == [1, -3, 127, -127, 0, 2, 0]
    q = orc.quantize_act(E4M3, x, np.float32(0.5))
    # 2, -6, 600 -> 448, -2e4 -> -448, 1, 3, -0
    assert list(q[0]) == [0x40, 0xCC, 0x7E, 0xFE, 0x38, 0x44, 0x80]


def test_calibrated_max_maps_to_qmax(orc):
    rng = np.random.default_rng(3)
    cal = synth.activations(512, 64, rng)
    for qt, top in ((INT8, 127), (E4M3, 0x7E)):
        s = orc.act_scale(qt, cal)
        q = orc.quantize_act(qt, cal, s)
        xf = synth.bf16_bits_to_f32(cal)
        i = np.unravel_index(np.abs(xf).argmax(), xf.shape)
        if qt == INT8:
            assert abs(int(q[i].view(np.int8))) == top
            assert np.abs(q.view(np.int8)).max() == 127
        else:
            assert (q[i] & 0x7F) == top


# ------------------------------------------------------------------- GEMMs
def test_i8_gemm_bruteforce_and_worst_case(orc):
    rng = np.random.default_rng(9)
    qx = rng.integers(-127, 128, (3, 37), dtype=np.int8)
    qw = rng.integers(-127, 128, (5, 37), dtype=np.int8)
    acc = orc.i8_gemm(qx, qw)
    for m in range(3):
        for n in range(5):
            assert acc[m, n] == sum(int(a) * int(b) for a, b in zip(qx[m], qw[n]))
    K = 18944
    ones = np.full((2, K), 127, np.int8)
    ones[1] = -127
    acc = orc.i8_gemm(ones, np.full((1, K), 127, np.int8))
    assert acc[0, 0] == 127 * 127 * K and acc[1, 0] == -127 * 127 * K


def test_i8_gemm_one_hot_selects_column(orc):
    rng = np.random.default_rng(2)
    K, N = 64, 16
    qx = rng.integers(-127, 128, (4, K), dtype=np.int8)
    perm = rng.permutation(K)[:N]
    qw = np.zeros((N, K), np.int8)
    qw[np.arange(N), perm] = 127
    acc = orc.i8_gemm(qx, qw)
    assert np.array_equal(acc, 127 * qx[:, perm].astype(np.int32))


def _hand_cases():
    cases = []
    for line in open(os.path.join(GOLDEN, "linear_hand.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        kind, rest = line.split(None, 1)
        fields = {}
        for part in rest.split("|"):
            toks = part.split()
            fields[toks[0]] = None if toks[1:] == ["-"] else [_num(t) for t in toks[1:]]
        cases.append((kind, fields))
    return cases


def test_hand_worked_linears(orc):
    for kind, f in _hand_cases():
        bias = None if f["b"] is None else synth.f32_to_bf16_bits(np.array(f["b"], np.float32))
        s_w = np.array(f["s"], np.float32)
        N = len(s_w)
        if kind.startswith("w8a16"):
            qt = INT8 if kind.endswith("int8") else E4M3
            K = len(f["q"]) // N
            x = synth.f32_to_bf16_bits(np.array(f["x"], np.float32).reshape(-1, K))
            q = np.array([int(v) & 0xFF for v in f["q"]], np.uint8).reshape(N, K)
            y = orc.w8a16(qt, x, q, s_w, bias)
        else:
            qt = INT8 if kind.endswith("int8") else E4M3
            K = len(f["qw"]) // N
            qx = np.array([int(v) & 0xFF for v in f["qx"]], np.uint8).reshape(-1, K)
            qw = np.array([int(v) & 0xFF for v in f["qw"]], np.uint8).reshape(N, K)
            y = orc.w8a8(qt, qx, np.float32(f["sx"][0]), qw, s_w, bias)
            if qt == INT8:
                assert list(orc.i8_gemm(qx, qw).ravel()) == [int(v) for v in f["acc"]]
        assert list(y.ravel()) == f["y"], (kind, y.ravel(), f["y"])


def _exact_deq(qt, c, orc):
    return Fraction(int(np.uint8(c).view(np.int8))) if qt == INT8 else Fraction(orc.e4m3_decode(int(c)))


@pytest.mark.parametrize("qt", [INT8, E4M3])
def test_w8a16_matches_exact_rationals(orc, qt):
    rng = np.random.default_rng(21 + qt)
    M, K, N = 3, 32, 5
    x = synth.activations(M, K, rng)
    w = synth.weights(N, K, rng)
    q, s = orc.quantize_weight(qt, w)
    b = synth.bias(N, rng)
    y = orc.w8a16(qt, x, q, s, b)
    xf = synth.bf16_bits_to_f32(x)
    bf = synth.bf16_bits_to_f32(b)
    for m in range(M):
        for n in range(N):
            acc = sum(Fraction(float(xf[m, k])) * _exact_deq(qt, q[n, k], orc) for k in range(K))
            ref = Fraction(float(s[n])) * acc + Fraction(float(bf[n]))
            assert abs(Fraction(y[m, n]) - ref) <= abs(ref) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)


@pytest.mark.parametrize("qt", [INT8, E4M3])
def test_w8a8_matches_exact_rationals(orc, qt):
    rng = np.random.default_rng(31 + qt)
    M, K, N = 2, 48, 4
    x = synth.activations(M, K, rng)
    s_x = orc.act_scale(qt, x)
    qx = orc.quantize_act(qt, x, s_x)
    q, s = orc.quantize_weight(qt, synth.weights(N, K, rng))
    b = synth.bias(N, rng)
    y = orc.w8a8(qt, qx, s_x, q, s, b)
    bf = synth.bf16_bits_to_f32(b)
    for m in range(M):
        for n in range(N):
            acc = sum(_exact_deq(qt, qx[m, k], orc) * _exact_deq(qt, q[n, k], orc) for k in range(K))
            ref = acc * Fraction(float(s_x)) * Fraction(float(s[n])) + Fraction(float(bf[n]))
            assert abs(Fraction(y[m, n]) - ref) <= abs(ref) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)


@pytest.mark.parametrize("qt", [INT8, E4M3])
def test_linearity_in_scales(orc, qt):
    """W * 2^j leaves the codes unchanged and scales s_w (and y) by exactly 2^j;
    x * 2^j does the same for the W8A8 activation path."""
    rng = np.random.default_rng(41)
    M, K, N = 4, 64, 8
    w = synth.weights(N, K, rng)
    x = synth.activations(M, K, rng)
    q1, s1 = orc.quantize_weight(qt, w)
    q2, s2 = orc.quantize_weight(qt, w * np.float32(8.0))
    assert np.array_equal(q1, q2) and np.array_equal(s2, s1 * np.float32(8.0))
    y1 = orc.w8a16(qt, x, q1, s1)
    y2 = orc.w8a16(qt, x, q2, s2)
    assert np.array_equal(y2, 8.0 * y1)
    x4 = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x) * np.float32(4.0))
    sa, sb = orc.act_scale(qt, x), orc.act_scale(qt, x4)
    assert sb == sa * np.float32(4.0)
    assert np.array_equal(orc.quantize_act(qt, x, sa), orc.quantize_act(qt, x4, sb))
    ya = orc.w8a8(qt, orc.quantize_act(qt, x, sa), sa, q1, s1)
    yb = orc.w8a8(qt, orc.quantize_act(qt, x4, sb), sb, q1, s1)
    assert np.array_equal(yb, 4.0 * ya)


def test_zero_weight_gives_bias(orc):
    rng = np.random.default_rng(1)
    K, N = 32, 16
    b = synth.bias(N, rng)
    x = synth.activations(3, K, rng)
    for qt in (INT8, E4M3):
        q, s = orc.quantize_weight(qt, np.zeros((N, K), np.float32))
        assert np.all(s == 1.0)
        y = orc.w8a16(qt, x, q, s, b)
        assert np.array_equal(y, np.broadcast_to(synth.bf16_bits_to_f32(b).astype(np.float64), y.shape))
        qx = orc.quantize_act(qt, x, orc.act_scale(qt, x))
        y = orc.w8a8(qt, qx, np.float32(0.37), q, s, b)
        assert np.array_equal(y, np.broadcast_to(synth.bf16_bits_to_f32(b).astype(np.float64), y.shape))


def test_row_sampling_consistent(orc):
    rng = np.random.default_rng(8)
    M, K, N = 10, 32, 6
    x = synth.activations(M, K, rng)
    q, s = orc.quantize_weight(E4M3, synth.weights(N, K, rng))
    full = orc.w8a16(E4M3, x, q, s)
    rows = [7, 0, 3]
    assert np.array_equal(orc.w8a16(E4M3, x, q, s, rows=rows), full[rows])
    qx = orc.quantize_act(E4M3, x, np.float32(0.01))
    full = orc.w8a8(E4M3, qx, 0.01, q, s)
    assert np.array_equal(orc.w8a8(E4M3, qx, 0.01, q, s, rows=rows), full[rows])


def test_quantizers_use_ieee_division(orc):
    """x/s is one correctly rounded binary32 division, not x * (1/s).  Rows are
    built with elements at and next to the rounding midpoints (k + 1/2 for INT8,
    midpoints of the E4M3 grid) times the row scale; there the two forms give
    different codes for some elements.  The test requires that such elements
    exist and that the oracle follows the division on every element."""
    rng = np.random.default_rng(1234)
    e4 = np.array([orc.e4m3_decode(c) for c in range(0x7F)])
    mids = {INT8: np.arange(-126, 127, dtype=np.float64) + 0.5,
            E4M3: np.concatenate([(e4[:-1] + e4[1:]) / 2, -(e4[:-1] + e4[1:]) / 2])}
    for qt, qmax in ((INT8, np.float32(127)), (E4M3, np.float32(448))):
        rows = []
        for _ in range(64):
            amax = np.float32(rng.uniform(0.01, 2.0))
            s = amax / qmax
            base = (mids[qt] * np.float64(s)).astype(np.float32)
            row = np.concatenate([[amax], base, np.nextafter(base, np.float32(np.inf)),
                                  np.nextafter(base, np.float32(-np.inf))]).astype(np.float32)
            rows.append(np.clip(row, -amax, amax))
        w = np.stack(rows)
        q, s = orc.quantize_weight(qt, w)
        assert np.array_equal(s, np.abs(w).max(axis=1) / qmax)
        v_div = w / s[:, None]
        v_rcp = w * (np.float32(1) / s)[:, None]
        if qt == INT8:
            def code(v):
                return np.clip(np.rint(v), -127, 127).astype(np.int8).view(np.uint8)
        else:
            def code(v):
                return torch.from_numpy(np.clip(v, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        c_div, c_rcp = code(v_div), code(v_rcp)
        assert (c_div != c_rcp).sum() >= 10, "no discriminating element in the sample"
        assert np.array_equal(q, c_div)


# ------------------------------------------- dynamic per-token activations
@pytest.mark.parametrize("qt", [INT8, E4M3])
def test_per_token_scales_and_extremes(orc, qt):
    rng = np.random.default_rng(61)
    x = synth.activations(9, 96, rng, synth.outlier_channels(96, rng))
    xf = synth.bf16_bits_to_f32(x)
    xf[3] = 0.0
    x = synth.f32_to_bf16_bits(xf)
    q, s = orc.quantize_act_per_token(qt, x)
    qmax = np.float32(127 if qt == INT8 else 448)
    for m in range(9):
        amax = np.abs(xf[m]).max()
        assert s[m] == (amax / qmax if amax > 0 else np.float32(1.0))
        if amax > 0:
            j = np.abs(xf[m]).argmax()
            code = q[m, j]
            assert (abs(int(code.view(np.int8))) == 127) if qt == INT8 else ((code & 0x7F) == 0x7E)
    assert np.all(q[3] == 0) and s[3] == 1.0


@pytest.mark.parametrize("qt", [INT8, E4M3])
def test_per_token_equals_static_when_rows_share_amax(orc, qt):
    """Rows with the same abs-max: the per-token quantizer reduces to the static
    one with that abs-max as calibration maximum."""
    rng = np.random.default_rng(62)
    xf = rng.standard_normal((7, 64)).astype(np.float32)
    xf[:, 5] = 6.0  # every row's largest magnitude
    x = synth.f32_to_bf16_bits(xf)
    q, s = orc.quantize_act_per_token(qt, x)
    s_static = orc.act_scale(qt, x)
    assert np.all(s == s_static)
    assert np.array_equal(q, orc.quantize_act(qt, x, s_static))


@pytest.mark.parametrize("qt", [INT8, E4M3])
def test_per_token_row_scaling_and_reference(orc, qt):
    """Scaling one token row by 2^j changes only that row's scale (by 2^j) and
    leaves every code and the W8A8 output of the other rows unchanged; the row's
    own output scales exactly.  The reference matches exact rationals."""
    rng = np.random.default_rng(63)
    M, K, N = 5, 48, 6
    xf = synth.bf16_bits_to_f32(synth.activations(M, K, rng))
    q1, s1 = orc.quantize_act_per_token(qt, synth.f32_to_bf16_bits(xf))
    xf2 = xf.copy()
    xf2[2] *= np.float32(8)
    q2, s2 = orc.quantize_act_per_token(qt, synth.f32_to_bf16_bits(xf2))
    assert np.array_equal(q1, q2)
    assert s2[2] == s1[2] * 8 and np.array_equal(np.delete(s1, 2), np.delete(s2, 2))
    qw, sw = orc.quantize_weight(qt, synth.weights(N, K, rng))
    b = synth.bias(N, rng)
    y1 = orc.w8a8_per_token(qt, q1, s1, qw, sw, b)
    y2 = orc.w8a8_per_token(qt, q2, s2, qw, sw)
    y1nb = orc.w8a8_per_token(qt, q1, s1, qw, sw)
    assert np.array_equal(y2[2], 8 * y1nb[2]) and np.array_equal(np.delete(y2, 2, 0), np.delete(y1nb, 2, 0))
    bf = synth.bf16_bits_to_f32(b)
    for m in range(M):
        for n in range(N):
            acc = sum(_exact_deq(qt, q1[m, k], orc) * _exact_deq(qt, qw[n, k], orc) for k in range(K))
            ref = acc * Fraction(float(s1[m])) * Fraction(float(sw[n])) + Fraction(float(bf[n]))
            assert abs(Fraction(y1[m, n]) - ref) <= abs(ref) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)
