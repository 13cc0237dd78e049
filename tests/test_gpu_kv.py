"""Mixed KV-cache kernels against the oracle, bit for bit (GPU).

qlin_kv_store_mixed writes INT8 key codes with float16 group-32 scales and E4M3
value codes with float16 per-(token, head) scales into a slot-addressed cache;
qlin_kv_load_mixed reads slots back as BF16.  Every output is an integer, a
float16 bit pattern or a BF16 rounding of an exact product, so all of them are
compared exactly, including the cache bytes the store must leave untouched.
"""
import numpy as np
import pytest
import torch

from bit_quantized_linear_gb300 import synth

pytestmark = pytest.mark.gpu
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def capi():
    from bit_quantized_linear_gb300 import capi as c
    return c


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _host_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _host_u8(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def _inputs(T, H, D, tag, ld_extra=0):
    """Token rows [T, H*D + ld_extra] with outlier channels, plus special rows: an
    all-zero token, a token with one zero key group and one zero value head, a tiny
    token (scales underflow float16), a huge token (scales saturate at 65504) and
    negative zeros."""
    rng = synth.rng_for("test-kv", 0, f"{T}x{H}x{D}", tag)
    outl = synth.outlier_channels(H * D, rng)
    k = synth.activations(T, H * D + ld_extra, rng, np.concatenate([outl, outl + 1]) % (H * D))
    v = synth.activations(T, H * D + ld_extra, rng, outl)
    special = [(0, lambda a: a * 0.0), (1, lambda a: a * 2.0 ** -140), (2, lambda a: a * 1.0e7),
               (3, lambda a: -np.abs(a) * 0.0)]
    for t, f in special:
        if t < T:
            for arr in (k, v):
                f32 = synth.bf16_bits_to_f32(arr[t]).astype(np.float64)
                arr[t] = synth.f32_to_bf16_bits(f(f32).astype(np.float32))
    if T > 4:
        k[4, 32:64] = 0
        v[4, :D] = 0
    return k, v


def _slots(T, num_slots, tag, pad_every=7):
    rng = synth.rng_for("test-kv-slots", 0, f"{T}/{num_slots}", tag)
    s = rng.permutation(num_slots)[:T].astype(np.int64)
    s[::pad_every] = -1
    return s


def _gpu_cache(capi, S, H, D):
    c = capi.kv_cache_alloc(S, H, D)
    for a in c:
        a.view(torch.uint8).fill_(SENTINEL)
    return c


def _compare_cache(gc, oc):
    np.testing.assert_array_equal(_host_u8(gc[0]), oc.k_cache)
    np.testing.assert_array_equal(_host_u16(gc[1]), oc.k_scale)
    np.testing.assert_array_equal(_host_u8(gc[2]), oc.v_cache)
    np.testing.assert_array_equal(_host_u16(gc[3]), oc.v_scale)


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("H,T", [(1, 1), (2, 37), (3, 64), (4, 300), (5, 33), (6, 129), (8, 1029)])
def test_kv_store_and_load_bit_exact(capi, orc, D, H, T):
    S = T + 64
    k, v = _inputs(T, H, D, "a")
    slots = _slots(T, S, "a")
    oc = orc.KVCache(S, H, D, fill=SENTINEL)
    assert orc.kv_store(oc, k, v, slots) == 0
    gc = _gpu_cache(capi, S, H, D)
    sl = torch.from_numpy(slots).cuda()
    capi.qlin_kv_store_mixed(_dev_bf16(k), _dev_bf16(v), sl, *gc)
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    _compare_cache(gc, oc)
    # read back every slot that was written, padding, and never-written slots (whose
    # sentinel bytes are valid codes and float16 scales on both sides)
    rng = np.random.default_rng(T * 7 + D)
    read = np.concatenate([slots, rng.integers(0, S, 40), [-1, -5]]).astype(np.int64)
    read = read[rng.permutation(read.size)]
    ko, vo, bad = orc.kv_load(oc, read)
    assert bad == 0
    gk, gv = capi.kv_load_mixed(torch.from_numpy(read).cuda(), gc)
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    np.testing.assert_array_equal(_host_u16(gk), ko)
    np.testing.assert_array_equal(_host_u16(gv), vo)


def test_kv_store_reads_strided_qkv_columns(capi, orc):
    """k and v passed in place as column ranges of a fused QKV output
    [T, (Hq + 2*Hkv) * D] (row stride (Hq + 2*Hkv) * D elements)."""
    T, Hq, H, D = 211, 28, 4, 128
    rng = synth.rng_for("test-kv", 0, "qkv", "strided")
    qkv = synth.activations(T, (Hq + 2 * H) * D, rng)
    k = qkv[:, Hq * D:(Hq + H) * D]
    v = qkv[:, (Hq + H) * D:]
    S = 512
    slots = _slots(T, S, "qkv")
    oc = orc.KVCache(S, H, D, fill=SENTINEL)
    orc.kv_store(oc, np.ascontiguousarray(k), np.ascontiguousarray(v), slots)
    gc = _gpu_cache(capi, S, H, D)
    dq = _dev_bf16(qkv)
    capi.qlin_kv_store_mixed(dq[:, Hq * D:(Hq + H) * D], dq[:, (Hq + H) * D:], torch.from_numpy(slots).cuda(), *gc)
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    _compare_cache(gc, oc)


def test_kv_full_size_7b_chunk(capi, orc):
    """The benchmark's shape: Qwen2.5-7B KV heads (H=4, D=128), an 8192-token prefill
    chunk scattered into 256-token blocks of a 32768-slot cache, then a 32768-token
    context read back; every byte compared."""
    H, D, block = 4, 128, 256
    S = 128 * block
    T = 8192
    k, v = _inputs(T, H, D, "full")
    rng = synth.rng_for("test-kv-slots", 0, "full", "blocks")
    blocks = rng.permutation(S // block)
    slots = (blocks[:T // block, None] * block + np.arange(block)[None, :]).reshape(-1).astype(np.int64)
    oc = orc.KVCache(S, H, D, fill=SENTINEL)
    orc.kv_store(oc, k, v, slots)
    gc = _gpu_cache(capi, S, H, D)
    capi.qlin_kv_store_mixed(_dev_bf16(k), _dev_bf16(v), torch.from_numpy(slots).cuda(), *gc)
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    _compare_cache(gc, oc)
    ctx = np.concatenate([slots, np.full(S - T, -1)]).astype(np.int64)
    ko, vo, _ = orc.kv_load(oc, ctx)
    gk, gv = capi.kv_load_mixed(torch.from_numpy(ctx).cuda(), gc)
    np.testing.assert_array_equal(_host_u16(gk), ko)
    np.testing.assert_array_equal(_host_u16(gv), vo)


def test_kv_out_of_range_slots_flagged_and_skipped(capi, orc):
    T, H, D, S = 40, 2, 64, 50
    k, v = _inputs(T, H, D, "oob")
    slots = _slots(T, S, "oob")
    slots[5] = S + 3
    slots[9] = S
    oc = orc.KVCache(S, H, D, fill=SENTINEL)
    assert orc.kv_store(oc, k, v, slots) == 2
    gc = _gpu_cache(capi, S, H, D)
    capi.qlin_kv_store_mixed(_dev_bf16(k), _dev_bf16(v), torch.from_numpy(slots).cuda(), *gc)
    assert capi.qlin_get_device_status() == capi.QLIN_ERR_INVALID_ARG
    assert capi.qlin_get_device_status() == capi.QLIN_OK  # reading clears it
    _compare_cache(gc, oc)
    read = np.array([slots[0] if slots[0] >= 0 else slots[1], S + 1, -1], np.int64)
    ko, vo, bad = orc.kv_load(oc, read)
    assert bad == 1
    gk, gv = capi.kv_load_mixed(torch.from_numpy(read).cuda(), gc)
    assert capi.qlin_get_device_status() == capi.QLIN_ERR_INVALID_ARG
    np.testing.assert_array_equal(_host_u16(gk), ko)
    np.testing.assert_array_equal(_host_u16(gv), vo)


def test_kv_zero_tokens_enqueue_nothing(capi):
    H, D, S = 4, 128, 16
    gc = _gpu_cache(capi, S, H, D)
    empty = torch.empty((0, H * D), dtype=torch.bfloat16, device="cuda")
    n0 = capi.qlin_launch_count()
    capi.qlin_kv_store_mixed(empty, empty, torch.empty(0, dtype=torch.int64, device="cuda"), *gc)
    k, v = capi.kv_load_mixed(torch.empty(0, dtype=torch.int64, device="cuda"), gc)
    assert capi.qlin_launch_count() == n0 and k.shape == (0, H, D)
    assert (_host_u8(gc[0]) == SENTINEL).all()
