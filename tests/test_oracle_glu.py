"""Pins for the oracle's merged gate_up linear with the SiLU * up epilogue (not gpu).

y[m, n] = silu(g) * u with g, u the linear's outputs for gate row n and up row
I + n of the merged weight [2I, K].  Pins: hand-worked cases
(tests/golden/glu_hand.txt), the identity silu(g) - silu(-g) = g (negating the
gate codes negates g exactly), equivariance under a joint permutation of the
gate and up rows, and the asymptotes silu(g) -> g and -> 0.
"""
import math
import os

import numpy as np
import pytest

from bit_quantized_linear_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
INT8, E4M3 = 0, 1


def _bf16(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, np.float32))


def _cases():
    out = []
    for line in open(os.path.join(GOLDEN, "glu_hand.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        kind, rest = line.split(None, 1)
        f = {}
        for part in rest.split("|"):
            name, *vals = part.split()
            f[name] = vals
        out.append((kind, f))
    return out


def test_glu_golden(orc):
    cases = _cases()
    assert len(cases) == 3
    for kind, f in cases:
        want = float(f["y"][0])
        s = np.array([float(v) for v in f["s"]], np.float32)
        b = None if f["b"] == ["-"] else _bf16([float(v) for v in f["b"]])
        if kind == "w8a16_int8":
            x = _bf16([[float(v) for v in f["x"]]])
            q = np.array([int(v) for v in f["q"]], np.int64).astype(np.int8).view(np.uint8).reshape(2, -1)
            y = orc.w8a16_gate_up_silu(INT8, x, q, s, b)
        else:
            qx = np.array([[int(v, 16) for v in f["qx"]]], np.uint8)
            q = np.array([int(v, 16) for v in f["q"]], np.uint8).reshape(2, -1)
            y = orc.w8a8_gate_up_silu(E4M3, qx, float(f["sx"][0]), q, s, b)
        assert y.shape == (1, 1)
        assert math.isclose(y[0, 0], want, rel_tol=1e-14), (kind, y[0, 0], want)


def _layer(qt, M, K, I, seed):
    rng = synth.rng_for("oracle-glu", 0, f"{M}x{K}x{I}", str(seed))
    w = synth.weights(2 * I, K, rng)
    x = synth.activations(M, K, rng)
    return w, x


def _negate_codes(qt, q):
    if qt == INT8:
        return (-(q.view(np.int8).astype(np.int16))).astype(np.int8).view(np.uint8)
    return q ^ np.uint8(0x80)


@pytest.mark.parametrize("qt", [INT8, E4M3])
def test_glu_silu_identity_and_pairing(orc, qt):
    """With the up rows' codes zero and the up bias 1, u = 1 and y = silu(g).  Negating
    the gate codes negates g exactly, and silu(g) - silu(-g) = g, where g is the plain
    linear's gate output.  Then a joint permutation of gate and up rows permutes y."""
    M, K, I = 5, 96, 24
    w, x = _layer(qt, M, K, I, 0)
    q, s = orc.quantize_weight(qt, w)
    q[I:] = 0
    bias = np.zeros(2 * I, np.uint16)
    bias[I:] = _bf16(np.ones(I))
    y_pos = orc.w8a16_gate_up_silu(qt, x, q, s, bias)
    qn = q.copy()
    qn[:I] = _negate_codes(qt, q[:I])
    y_neg = orc.w8a16_gate_up_silu(qt, x, qn, s, bias)
    g = orc.w8a16(qt, x, q[:I], s[:I])
    np.testing.assert_allclose(y_pos - y_neg, g, rtol=1e-12, atol=1e-12 * np.abs(g).max())
    # joint permutation of (gate row n, up row I + n) permutes the output columns
    w2, _ = _layer(qt, M, K, I, 1)
    q2, s2 = orc.quantize_weight(qt, w2)
    y = orc.w8a16_gate_up_silu(qt, x, q2, s2)
    perm = np.random.default_rng(3).permutation(I)
    rows = np.concatenate([perm, I + perm])
    yp = orc.w8a16_gate_up_silu(qt, x, q2[rows], s2[rows])
    np.testing.assert_array_equal(yp, y[:, perm])
    # gate and up do not commute: swapping the halves changes the result
    sw = np.concatenate([np.arange(I, 2 * I), np.arange(I)])
    assert not np.allclose(orc.w8a16_gate_up_silu(qt, x, q2[sw], s2[sw]), y)


def test_glu_asymptotes_and_w8a8(orc):
    """silu(g) -> g for large g and -> 0 for very negative g (u = 2 via the up bias);
    the W8A8 form follows the same definition on the W8A8 linear."""
    K, I = 32, 2
    x = _bf16([[1.0] * K])
    q = np.zeros((2 * I, K), np.uint8)
    q[0, :] = 127            # g = 127 * K * s
    q[1, :] = np.uint8(0x81)  # -127
    s = np.array([0.05, 0.05, 1.0, 1.0], np.float32)
    bias = _bf16([0, 0, 2.0, 2.0])
    y = orc.w8a16_gate_up_silu(INT8, x, q, s, bias)
    g = 127 * K * np.float64(np.float32(0.05))
    assert math.isclose(y[0, 0], 2 * g, rel_tol=1e-12) and 0.0 >= y[0, 1] > -1e-50
    qx = np.full((1, K), 0x38, np.uint8)  # E4M3 1.0
    qe = np.zeros((2 * I, K), np.uint8)
    qe[0, :] = 0x38
    qe[1, :] = 0xB8  # -1
    ye = orc.w8a8_gate_up_silu(E4M3, qx, 0.25, qe, np.ones(2 * I, np.float32), bias)
    lin = orc.w8a8(E4M3, qx, 0.25, qe, np.ones(2 * I, np.float32), bias)
    # silu(8) * 2 and silu(-8) * 2 from the linear's own outputs
    assert math.isclose(ye[0, 0] / lin[0, 2], lin[0, 0] / (1 + math.exp(-lin[0, 0])), rel_tol=1e-14)
    assert math.isclose(ye[0, 1] / lin[0, 3], lin[0, 1] / (1 + math.exp(-lin[0, 1])), rel_tol=1e-14)
