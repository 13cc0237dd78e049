"""The quantizers' quotient x / s against the oracle's IEEE division (GPU).

The kernels divide by a scale shared by a whole row, group or tensor, so they
compute x / s from the correctly rounded reciprocal with one FMA correction
(Markstein's theorem) instead of a division per element.  These tests sweep
every finite BF16 value through each quantizer over many scales, including
the edges of the fast path's scale range, and require bit-identical codes with
the oracle.  Each also checks that its sample contains elements where a plain
reciprocal multiply x * (1/s) would give a different code, so that a quotient
one ulp off at a rounding boundary cannot pass.
"""
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


def _all_bf16():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    return bits[np.isfinite(synth.bf16_bits_to_f32(bits))]


def _code_np(qt, v):
    if qt == "int8":
        return np.clip(np.rint(v), -127, 127).astype(np.int8).view(np.uint8)
    return torch.from_numpy(np.clip(v, -448, 448).astype(np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def _e4m3_midpoints():
    e4 = torch.arange(0x7F, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    return (e4[:-1] + e4[1:]) / 2


def _search_amax(qt, scale_of, n, seed, keep=16):
    """BF16 abs-max values whose scale gives discriminating elements among the BF16
    values below them (random candidates, plain search)."""
    allb = _all_bf16()
    allf = synth.bf16_bits_to_f32(allb)
    pos = allb[(allf > 1e-4) & (allf < 1e5)]
    rng = np.random.default_rng(seed)
    out = []
    for ab in rng.choice(pos, min(n, len(pos)), replace=False):
        a = synth.bf16_bits_to_f32(np.array([ab]))[0]
        if _discriminating(qt, allb[np.abs(allf) < a], scale_of(a)):
            out.append(float(a))
            if len(out) == keep:
                break
    return out


def _discriminating(qt, x_bits, s):
    """Elements whose code differs between x / s and x * RN(1/s) (numpy float32)."""
    x = synth.bf16_bits_to_f32(x_bits)
    s = np.float32(s)
    with np.errstate(over="ignore", invalid="ignore"):
        return int((_code_np(qt, x / s) != _code_np(qt, x * (np.float32(1) / s))).sum())


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_static_quantizer_all_bf16_many_scales(capi, qt):
    bits = _all_bf16()
    bits = np.concatenate([bits, np.zeros((-len(bits)) % 16, np.uint16)]).reshape(-1, 16)
    rng = np.random.default_rng(11)
    scales = [np.float32(2.0 ** e) for e in (-97, -96, -20, 0, 20, 96, 97)]
    scales += list((2.0 ** rng.uniform(-30, 30, 60)).astype(np.float32))
    # scales that put some BF16 value x0 on a rounding midpoint m of the code grid
    allf = synth.bf16_bits_to_f32(_all_bf16())
    x0s = rng.choice(allf[(allf > 1e-6) & (allf < 1e6)], 60)
    mids = (np.arange(0, 127) + 0.5) if qt == "int8" else _e4m3_midpoints()
    scales += [np.float32(np.float32(x0) / np.float32(m)) for x0, m in zip(x0s, rng.choice(mids[mids > 0], 60))]
    disc = 0
    xd = to_dev_bf16(bits)
    for s in scales:
        qx = capi.quantize_act_static(qt, xd, to_dev(np.array([s], np.float32))).cpu().numpy()
        oq = oracle.quantize_act(QT[qt], bits, s)
        bad = np.nonzero(qx != oq)
        assert bad[0].size == 0, (qt, float(s), bad[0].size, hex(bits[bad][0]))
        disc += _discriminating(qt, bits.reshape(-1), s)
    assert disc >= 3, disc


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_dynamic_quantizer_all_bf16_below_row_max(capi, qt):
    """Rows whose first element sets the row's abs-max and whose other elements are
    every BF16 value of smaller magnitude."""
    allb = _all_bf16()
    allf = synth.bf16_bits_to_f32(allb)
    qmax = np.float32(127 if qt == "int8" else 448)
    found = _search_amax(qt, lambda a: np.float32(a) / qmax, 3000, 12)
    amaxes = np.concatenate([[1.0, 448.0, 127.0, 2.0 ** -20, 3.0e4], found])
    rows = []
    for a in amaxes:
        ab = synth.f32_to_bf16_bits(np.array([a], np.float32))[0]
        af = synth.bf16_bits_to_f32(np.array([ab]))[0]
        vals = allb[np.abs(allf) < af]
        rows.append(np.concatenate([[ab], vals]))
    K = max(len(r) for r in rows)
    K += (-K) % 16
    x = np.zeros((len(rows), K), np.uint16)
    for i, r in enumerate(rows):
        x[i, :len(r)] = r
    qx, sx = capi.quantize_act_dynamic(qt, to_dev_bf16(x))
    oq, os_ = oracle.quantize_act_per_token(QT[qt], x)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    qx = qx.cpu().numpy()
    bad = np.nonzero(qx != oq)
    assert bad[0].size == 0, (bad[0].size, bad[0][0], hex(x[bad][0]))
    disc = sum(_discriminating(qt, x[i], os_[i]) for i in range(len(rows)))
    assert disc >= 3, disc


def test_kv_store_all_bf16_below_group_max(capi):
    """Key groups / value heads of 32 elements (H=1, D=32): element 0 sets the
    abs-max, the other 31 walk through every BF16 value of smaller magnitude."""
    allb = _all_bf16()
    allf = synth.bf16_bits_to_f32(allb)
    f16 = lambda a, q: np.float32(np.float16(np.float32(a) / np.float32(q)))
    found_k = _search_amax("int8", lambda a: f16(a, 127), 6000, 13, keep=12)
    found_v = _search_amax("e4m3", lambda a: f16(a, 448), 3000, 14, keep=12)
    amaxes = np.concatenate([[1.0, 127.0, 448.0, 2.0 ** -18, 6.0e4, 1.0e7], found_k, found_v])
    toks = []
    for a in amaxes:
        ab = synth.f32_to_bf16_bits(np.array([a], np.float32))[0]
        af = synth.bf16_bits_to_f32(np.array([ab]))[0]
        vals = allb[np.abs(allf) < af]
        vals = np.concatenate([vals, np.zeros((-len(vals)) % 31, np.uint16)]).reshape(-1, 31)
        toks.append(np.concatenate([np.full((len(vals), 1), ab, np.uint16), vals], axis=1))
    kv = np.concatenate(toks)
    T = kv.shape[0]
    slots = np.arange(T, dtype=np.int64)
    oc = oracle.KVCache(T, 1, 32)
    oracle.kv_store(oc, kv, kv, slots)
    gc = capi.kv_cache_alloc(T, 1, 32)
    xd = to_dev_bf16(kv)
    capi.qlin_kv_store_mixed(xd, xd, torch.from_numpy(slots).cuda(), *gc)
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    for g, o, name in ((gc[0].view(torch.uint8), oc.k_cache, "k codes"), (gc[2], oc.v_cache, "v codes")):
        got = g.cpu().numpy().reshape(o.shape)
        bad = np.nonzero(got != o)
        assert bad[0].size == 0, (name, bad[0].size, bad[0][0])
    assert np.array_equal(gc[1].cpu().numpy().view(np.uint16), oc.k_scale)
    assert np.array_equal(gc[3].cpu().numpy().view(np.uint16), oc.v_scale)
    ks = oc.k_scale.view(np.float16).astype(np.float32).reshape(-1)
    vs = oc.v_scale.view(np.float16).astype(np.float32).reshape(-1)
    assert sum(_discriminating("int8", kv[t], ks[t]) for t in range(T)) >= 1
    assert sum(_discriminating("e4m3", kv[t], vs[t]) for t in range(T)) >= 3
