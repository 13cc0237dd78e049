"""Shared test helpers: host<->device marshalling and the BF16 output tolerance.

Tolerance for BF16 outputs (the layer's stated bar): per element
|y - y_ref| <= 8e-3 * |y_ref| + 1e-3 * rms(y_ref), and relative Frobenius error
||y - y_ref||_F / ||y_ref||_F <= 2e-3, with y_ref the oracle's fp64 result.
"""
import numpy as np
import torch

ELEM_REL, ELEM_RMS, FRO = 8e-3, 1e-3, 2e-3


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def from_dev_bf16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(bits):
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_tol(y_bits, ref, what=""):
    """y_bits: BF16 bits from the device; ref: fp64 oracle values (same shape)."""
    y = bf16_to_f64(y_bits)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bound = ELEM_REL * np.abs(ref) + ELEM_RMS * rms
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"y={y[i]!r} ref={ref[i]!r} bound={bound[i]!r}")
    nref = np.linalg.norm(ref)
    fro = float(np.linalg.norm(y - ref) / nref) if nref > 0 else float(np.linalg.norm(y))
    assert fro <= FRO, f"{what}: relative Frobenius error {fro:.3e} > {FRO}"
    return fro


def sample_rows(M, n=16, seed=0):
    """Deterministic row sample covering the first and last rows."""
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, M - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, M - 1], mid]))
