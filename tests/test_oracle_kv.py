"""Pins for the oracle's mixed KV-cache quantizers (not gpu).

Keys are INT8 with one float16 scale per 32 head_dim elements, values E4M3
with one float16 scale per token and kv head ("Nano-vLLM-MoE" README, section
"KV cache compression").  The pins: hand-worked groups (tests/golden/kv_hand.txt),
the page's own byte counts (bytes per block and the 7B arena sizes), numpy's
float16 conversion and torch's BF16 conversion as independent casts, and
invariants that a wrong group boundary, head index or slot would break.
"""
import math
import os

import numpy as np
import pytest
import torch

from bit_quantized_linear_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(t):
    t = t.strip()
    if "p" in t.lower():
        return float.fromhex(t)
    return float(t)


def _bf16_bits_exact(v):
    """BF16 bits of a value that is exactly representable in BF16."""
    f = np.float32(v)
    assert float(f) == v or (math.isnan(v) and math.isnan(f))
    u = int(np.array([f], np.float32).view(np.uint32)[0])
    assert u & 0xFFFF == 0, v
    return u >> 16


def _kv_cases():
    out = []
    for line in open(os.path.join(GOLDEN, "kv_hand.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        kind, rest = line.split(None, 1)
        f = {}
        for part in rest.split("|"):
            name, *vals = part.split()
            f[name] = vals
        x = [_num(t) for t in f["x"]]
        scale = _num(f["scale"][0])
        if kind == "kgroup":
            q = [int(t) & 0xFF for t in f["q"]]
        else:
            q = [int(t, 16) for t in f["q"]]
        deq = [_num(t) for t in f["deq"]]
        out.append((kind, x, scale, q, deq))
    return out


def test_kv_golden_groups(orc):
    cases = _kv_cases()
    assert sum(c[0] == "kgroup" for c in cases) == 6 and sum(c[0] == "vhead" for c in cases) == 3
    for kind, x, scale, q, deq in cases:
        D = 32
        row = np.zeros((1, D), np.uint16)
        row[0, :len(x)] = [_bf16_bits_exact(v) for v in x]
        zero = np.zeros((1, D), np.uint16)
        c = orc.KVCache(3, 1, D, fill=0xA5)
        k_in, v_in = (row, zero) if kind == "kgroup" else (zero, row)
        assert orc.kv_store(c, k_in, v_in, [1]) == 0
        want_q = np.zeros(D, np.uint8)
        want_q[:len(q)] = q
        want_deq = np.zeros(D, np.uint16)
        want_deq[:len(deq)] = [_bf16_bits_exact(v) for v in deq]
        scale_bits = int(np.array([scale], np.float16).view(np.uint16)[0])
        assert float(np.float16(scale)) == scale
        ko, vo, bad = orc.kv_load(c, [1])
        assert bad == 0
        if kind == "kgroup":
            assert c.k_scale[1, 0, 0] == scale_bits, (x[:3], hex(c.k_scale[1, 0, 0]), hex(scale_bits))
            np.testing.assert_array_equal(c.k_cache[1, 0], want_q)
            np.testing.assert_array_equal(ko[0, 0], want_deq)
        else:
            assert c.v_scale[1, 0] == scale_bits, (x[:3], hex(c.v_scale[1, 0]), hex(scale_bits))
            np.testing.assert_array_equal(c.v_cache[1, 0], want_q)
            np.testing.assert_array_equal(vo[0, 0], want_deq)
        # untouched slots keep their contents
        assert (c.k_cache[[0, 2]] == 0xA5).all() and (c.v_scale[[0, 2]] == 0xA5A5).all()


def test_kv_layout_matches_page_byte_counts(orc):
    """The page prints 0.5195x BF16 bytes per block and a 7B arena of 512 blocks that
    shrinks from 7.00 GiB (BF16) to 3.64 GiB.  Qwen2.5-7B has 28 layers, 4 kv heads and
    head_dim 128; 512 blocks of 256 tokens reproduce the BF16 figure.  The layout read
    from the page (float16 scale per 32 key elements and per token-head for values)
    reproduces both numbers; a per-token value scale shared by all heads would not."""
    layers, H, D, blocks, block_size = 28, 4, 128, 512, 256
    c = orc.KVCache(block_size, H, D)
    per_block = c.nbytes()
    bf16_per_block = 2 * block_size * H * D * 2
    assert round(per_block / bf16_per_block, 4) == 0.5195
    gib = 1024 ** 3
    assert round(layers * blocks * bf16_per_block / gib, 2) == 7.00
    assert round(layers * blocks * per_block / gib, 2) == 3.64
    alt = per_block - block_size * (H - 1) * 2  # one value scale per token for all heads
    assert round(alt / bf16_per_block, 4) != 0.5195


# ------------------------------------------------------------ float16 / BF16 casts
def _finite_fp16_codes():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return h[(h & 0x7C00) != 0x7C00]


def test_fp16_decode_matches_numpy_all_codes(orc):
    codes = _finite_fp16_codes()
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([orc.fp16_decode(int(c)) for c in codes])
    np.testing.assert_array_equal(got, ref)
    assert math.copysign(1.0, orc.fp16_decode(0x8000)) == -1.0


def test_fp16_encode_roundtrip_and_midpoints(orc):
    codes = _finite_fp16_codes()
    for c in codes[::7]:
        assert orc.fp16_encode(orc.fp16_decode(int(c))) == int(c)
    pos = np.sort(codes[codes < 0x8000].view(np.float16).astype(np.float64))
    mids = (pos[:-1] + pos[1:]) / 2  # exact in fp64
    ref = mids.astype(np.float16).view(np.uint16)  # numpy: round half to even
    for m, r in zip(mids[::3], ref[::3]):
        assert orc.fp16_encode(float(m)) == int(r), (m, hex(orc.fp16_encode(float(m))), hex(int(r)))
        assert orc.fp16_encode(-float(m)) == int(r) | 0x8000


def test_fp16_encode_matches_numpy_random_and_saturates(orc):
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
                        rng.uniform(-65519, 65519, 500)])
    ref = v.astype(np.float16).view(np.uint16)
    for a, r in zip(v, ref):
        assert orc.fp16_encode(float(a)) == int(r), a
    for big in (65520.0, 7e4, 1e30):
        assert orc.fp16_encode(big) == 0x7BFF and orc.fp16_encode(-big) == 0xFBFF
    assert orc.fp16_encode(-0.0) == 0x8000 and orc.fp16_encode(2.0 ** -26) == 0


def test_bf16_encode_matches_torch(orc):
    rng = np.random.default_rng(6)
    v = (rng.standard_normal(6000) * 10.0 ** rng.integers(-30, 30, 6000)).astype(np.float32)
    f32_bits = v.view(np.uint32)
    mids = ((f32_bits & ~np.uint32(0xFFFF)) | np.uint32(0x8000)).view(np.float32)  # exact ties
    allv = np.concatenate([v, mids, np.float32([2.0 ** -130, -(2.0 ** -149), 3.0e38])])
    ref = torch.from_numpy(allv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for a, r in zip(allv, ref):
        assert orc.bf16_encode(float(a)) == int(r), (a, hex(orc.bf16_encode(float(a))), hex(int(r)))


# ------------------------------------------------------------ invariants
def _rand_kv(T, H, D, seed, ld_pad=0):
    rng = synth.rng_for("oracle-kv", 0, f"{T}x{H}x{D}", str(seed))
    k = synth.activations(T, H * D + ld_pad, rng)
    v = synth.activations(T, H * D + ld_pad, rng)
    return k, v


def _scale_bf16(bits, j):
    f = synth.bf16_bits_to_f32(bits).astype(np.float64) * 2.0 ** j
    return synth.f32_to_bf16_bits(f.astype(np.float32))


def test_kv_group_and_head_locality(orc):
    """Scaling one 32-element key group (or one value head) by 2^j changes exactly that
    group's (head's) float16 scale, by 2^j, and no code anywhere."""
    T, H, D = 3, 2, 128
    k, v = _rand_kv(T, H, D, 0)
    slots = np.array([5, 0, 3])
    base = orc.KVCache(8, H, D)
    orc.kv_store(base, k, v, slots)
    for (t, h, g, j) in [(0, 0, 0, 3), (1, 1, 3, -2), (2, 0, 2, 5), (2, 1, 1, -4)]:
        k2 = k.copy()
        sl = slice(h * D + 32 * g, h * D + 32 * g + 32)
        k2[t, sl] = _scale_bf16(k2[t, sl], j)
        c = orc.KVCache(8, H, D)
        orc.kv_store(c, k2, v, slots)
        np.testing.assert_array_equal(c.k_cache, base.k_cache)
        np.testing.assert_array_equal(c.v_cache, base.v_cache)
        np.testing.assert_array_equal(c.v_scale, base.v_scale)
        diff = np.argwhere(c.k_scale != base.k_scale)
        assert diff.tolist() == [[slots[t], h, g]]
        s0 = np.float64(base.k_scale[slots[t], h, g:g + 1].view(np.float16)[0])
        s1 = np.float64(c.k_scale[slots[t], h, g:g + 1].view(np.float16)[0])
        assert s1 == s0 * 2.0 ** j
        v2 = v.copy()
        v2[t, h * D:(h + 1) * D] = _scale_bf16(v2[t, h * D:(h + 1) * D], j)
        c = orc.KVCache(8, H, D)
        orc.kv_store(c, k, v2, slots)
        np.testing.assert_array_equal(c.k_cache, base.k_cache)
        np.testing.assert_array_equal(c.k_scale, base.k_scale)
        np.testing.assert_array_equal(c.v_cache, base.v_cache)
        assert np.argwhere(c.v_scale != base.v_scale).tolist() == [[slots[t], h]]


def test_kv_max_element_codes_and_scale_cast(orc):
    """The group (head) maximum maps to +-127 (+-448) and the float16 scale is within half a
    float16 step of amax/QMAX."""
    T, H, D = 6, 4, 64
    k, v = _rand_kv(T, H, D, 1)
    c = orc.KVCache(T, H, D)
    orc.kv_store(c, k, v, np.arange(T))
    kf = synth.bf16_bits_to_f32(k).reshape(T, H, D // 32, 32).astype(np.float64)
    vf = synth.bf16_bits_to_f32(v).reshape(T, H, D).astype(np.float64)
    kq = c.k_cache.view(np.int8).reshape(T, H, D // 32, 32)
    am = np.abs(kf).argmax(-1)
    assert (np.abs(np.take_along_axis(kq, am[..., None], -1)) == 127).all()
    ks = c.k_scale.view(np.float16).astype(np.float64)
    amax = np.abs(kf).max(-1)
    ulp = 2.0 ** (np.floor(np.log2(amax / 127)) - 10)
    assert (np.abs(ks - amax / 127) <= ulp / 2 * (1 + 1e-6)).all()
    vc = c.v_cache
    amv = np.abs(vf).argmax(-1)
    assert ((np.take_along_axis(vc, amv[..., None], -1) & 0x7F) == 0x7E).all()


def test_kv_roundtrip_error_bounds(orc):
    """load(store(x)) is within half a quantization step of x (plus one BF16 rounding)
    for keys, and within the E4M3 half-step for values."""
    T, H, D = 16, 2, 128
    k, v = _rand_kv(T, H, D, 2)
    c = orc.KVCache(40, H, D)
    slots = np.arange(T) * 2 + 1
    orc.kv_store(c, k, v, slots)
    ko, vo, bad = orc.kv_load(c, slots)
    assert bad == 0
    kf = synth.bf16_bits_to_f32(k).reshape(T, H, D).astype(np.float64)
    vf = synth.bf16_bits_to_f32(v).reshape(T, H, D).astype(np.float64)
    kd = synth.bf16_bits_to_f32(ko).astype(np.float64)
    vd = synth.bf16_bits_to_f32(vo).astype(np.float64)
    ks = np.repeat(c.k_scale[slots].view(np.float16).astype(np.float64), 32, axis=-1)
    assert (np.abs(kd - kf) <= ks / 2 + np.abs(kd) * 2.0 ** -8).all()
    vs = c.v_scale[slots].view(np.float16).astype(np.float64)[..., None]
    step = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(vf) / vs, 2.0 ** -6))) - 3), 2.0 ** -9) * vs
    assert (np.abs(vd - vf) <= step / 2 + np.abs(vd) * 2.0 ** -8).all()


def test_kv_store_scatter_and_load_padding(orc):
    """Tokens land in their own slots, negative slots are skipped on store and read as +0 on
    load, out-of-range slots are counted and skipped, and strided input rows read only the
    first H*D elements of each row."""
    T, H, D = 7, 2, 64
    k, v = _rand_kv(T, H, D, 3, ld_pad=24)
    slots = np.array([4, -1, 9, 0, 12, -1, 2])
    c = orc.KVCache(12, H, D, fill=0x5A)
    assert orc.kv_store(c, k, v, slots) == 1  # slot 12 >= num_slots
    written = {4, 9, 0, 2}
    for s in range(12):
        if s not in written:
            assert (c.k_cache[s] == 0x5A).all() and (c.k_scale[s] == 0x5A5A).all()
            assert (c.v_cache[s] == 0x5A).all() and (c.v_scale[s] == 0x5A5A).all()
    for t, s in enumerate(slots):
        if s in written:
            one = orc.KVCache(1, H, D)
            orc.kv_store(one, k[t:t + 1, :H * D].copy(), v[t:t + 1, :H * D].copy(), [0])
            for a, b in ((one.k_cache, c.k_cache), (one.k_scale, c.k_scale),
                         (one.v_cache, c.v_cache), (one.v_scale, c.v_scale)):
                np.testing.assert_array_equal(a[0], b[s])
    ko, vo, bad = orc.kv_load(c, [-1, 4, 12, 0])
    assert bad == 1
    assert (ko[[0, 2]] == 0).all() and (vo[[0, 2]] == 0).all()
    assert (ko[1] != 0).any() and (vo[3] != 0).any()
