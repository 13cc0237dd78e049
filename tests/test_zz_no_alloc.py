"""The allocation-free W8A8 entry point (GPU).

qlin_w8a8_linear_noalloc serves callers that cannot allocate device memory,
for example a plugin running inside an engine that owns all device memory, or
code enqueued while a stream is being captured into a CUDA graph.  It keeps its
quantized-activation scratch in a library-owned device array instead of a
caller workspace.  These tests call it through the C ABI and compare it with
the ordinary workspace-taking qlin_w8a8_linear on the same inputs, two calls in
a row (the second call finds the first call's data in the shared scratch), and
check that sizes beyond the scratch are refused before any launch.

This file is named to be collected last.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from bit_quantized_linear_gb300 import synth
from _helpers import bf16_to_f64, check_tol, from_dev_bf16

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def capi():
    from bit_quantized_linear_gb300 import capi as c
    return c


def _inputs(capi, qt, M, K, N, tag):
    rng = synth.rng_for("test-noalloc", 0, f"{qt}-{M}x{K}x{N}-{tag}", "all")
    outl = synth.outlier_channels(K, rng)
    dev = torch.device("cuda")
    w = torch.from_numpy(synth.weights(N, K, rng)).to(dev)
    cal = torch.from_numpy(synth.activations(2048, K, rng, outl).view(np.int16)).to(dev).view(torch.bfloat16)
    x = torch.from_numpy(synth.activations(M, K, rng, outl).view(np.int16)).to(dev).view(torch.bfloat16)
    b = torch.from_numpy(synth.bias(N, rng).view(np.int16)).to(dev).view(torch.bfloat16)
    qw, s = capi.quantize_weight(qt, w)
    sx = capi.act_scale_from_calib(qt, cal)
    return x, sx, qw, s, b


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_noalloc_matches_workspace_entry_point_twice(capi, qt):
    shapes = [(77, 1024, 384), (300, 2048, 272)]  # two calls in a row with different sizes
    for i, (M, K, N) in enumerate(shapes):
        x, sx, qw, s, b = _inputs(capi, qt, M, K, N, i)
        y_ref = capi.w8a8_linear(qt, x, sx, qw, s, b)
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        capi.qlin_w8a8_linear_noalloc(qt, x, sx, qw, s, b, y)
        torch.cuda.synchronize()
        assert capi.qlin_get_device_status() == capi.QLIN_OK
        check_tol(from_dev_bf16(y), bf16_to_f64(from_dev_bf16(y_ref)), f"noalloc {qt} call {i}")


def test_noalloc_rejects_sizes_beyond_scratch(capi):
    """The largest M whose workspace fits the scratch is accepted by the size
    check; one row more is refused with QLIN_ERR_WORKSPACE before any launch."""
    L = capi.lib()
    limit = capi.W8A8_NOALLOC_SCRATCH_BYTES
    src = open(os.path.join(ROOT, "include", "qlin.h")).read()
    assert re.search(r"QLIN_W8A8_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)32 << 20\)", src)
    K, N = 4096, 256
    p = ctypes.c_void_p(4096)  # never dereferenced: refused before any launch
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for qt in ("int8", "e4m3"):
        need = lambda M: capi.qlin_workspace_bytes(capi.QLIN_OP_W8A8_LINEAR, qt, M, K, N)
        lo, hi = 1, limit  # need() grows with M: the largest M whose workspace fits
        while lo < hi:
            mid = (lo + hi + 1) // 2
            lo, hi = (mid, hi) if need(mid) <= limit else (lo, mid - 1)
        m_max = lo
        assert need(m_max) <= limit < need(m_max + 1)
        st = L.qlin_w8a8_linear_noalloc(capi.QTYPES[qt], m_max + 1, K, N, p, p, p, p, None, p, stream)
        assert st == capi.QLIN_ERR_WORKSPACE
