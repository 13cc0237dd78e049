"""The arithmetic behind the E4M3 W8A16 path for small batches (not gpu).

Up to 32 tokens, E4M3 W8A16 multiplies the weight codes on the FP8 tensor
cores against the activations written as E4M3 terms.  Each element
v = x / s (s a power of two with 448 s >= max |x| of the row) goes into one of
two bands:
    band A, |v| >= 2^-6:  v = x1 + x2 / 16,
    band B, |v| <  2^-6:  v = 2^-14 (x3 + x4 / 16),
with x1 = RN(u), x2 = RN(16 (u - x1)) for the band's value u (v, or 2^14 v),
RN the round-to-nearest-even cast to OCP E4M3.  These tests check, over every
BF16 value, the claims the kernel's accuracy rests on: the split is exact for
|v| >= 2^-20, and below that its error is at most 2^-28 (in units of s).  The
cast is torch's float8_e4m3fn conversion, an implementation independent of
the CUDA path.
"""
import numpy as np
import torch


def _e4m3(a):
    """Round-to-nearest-even to E4M3 (values within +-448), back to float64."""
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def _split(v):
    """(x1, x2, x3, x4) of the two-band split of float32 values v, |v| <= 448."""
    v = np.asarray(v, np.float32)
    lo = np.abs(v) < np.float32(2.0 ** -6)
    u = np.where(lo, v * np.float32(16384.0), v).astype(np.float32)
    t1 = _e4m3(u)
    t2 = _e4m3((16.0 * (u.astype(np.float64) - t1)).astype(np.float32))
    z = np.zeros_like(t1)
    return np.where(lo, z, t1), np.where(lo, z, t2), np.where(lo, t1, z), np.where(lo, t2, z)


def _all_bf16_up_to(limit):
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # every finite non-negative BF16 value
    vals = (bits << 16).view(np.float32)
    vals = vals[vals <= limit]
    return np.concatenate([vals, -vals])


def _reconstruct(v):
    x1, x2, x3, x4 = _split(v)
    return x1 + x2 / 16.0 + 2.0 ** -14 * (x3 + x4 / 16.0)


def test_split_is_exact_from_2_pow_minus_20_up():
    v = _all_bf16_up_to(448.0)
    big = np.abs(v) >= 2.0 ** -20
    r = _reconstruct(v)
    assert np.array_equal(r[big], v[big].astype(np.float64))


def test_split_error_below_2_pow_minus_20_is_at_most_2_pow_minus_28():
    v = _all_bf16_up_to(448.0)
    small = np.abs(v) < 2.0 ** -20
    err = np.abs(_reconstruct(v)[small] - v[small].astype(np.float64))
    assert err.max() <= 2.0 ** -28


def test_terms_fit_e4m3_without_saturation():
    """No term reaches past 448 (no saturation), and band A holds exactly the
    elements with |v| >= 2^-6."""
    v = _all_bf16_up_to(448.0)
    x1, x2, x3, x4 = _split(v)
    for t in (x1, x2, x3, x4):
        assert np.abs(t).max() <= 448.0
    band_a = np.abs(v) >= 2.0 ** -6
    assert np.all((x3[band_a] == 0) & (x4[band_a] == 0))
    assert np.all((x1[~band_a] == 0) & (x2[~band_a] == 0))


def test_one_band_alone_would_lose_small_elements():
    """The reason for band B: with band A's terms alone, an element 2^-10 of the
    scale (a row whose maximum is 2^18 above its ordinary elements) keeps at
    most 2^-14 absolute precision, which loses most of its 8 bits."""
    v = np.float32(2.0 ** -10 * 1.6796875)  # a BF16 value with all 8 significant bits used
    t1 = _e4m3(v)
    t2 = _e4m3(np.float32(16.0 * (float(v) - float(t1[()]))))
    one_band = float(t1[()]) + float(t2[()]) / 16.0
    assert one_band != float(v)
    assert float(_reconstruct(np.array([v]))[0]) == float(v)
