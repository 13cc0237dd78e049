"""The allocation-free W8A8 entry point (GPU).

qlin_w8a8_linear_noalloc serves callers that cannot allocate device memory,
for example a plugin running inside an engine that owns all device memory, or
code enqueued while a stream is being captured into a CUDA graph.  It keeps its
quantized-activation scratch (and the task flags of the fused-quantization FP8
GEMM) in a library-owned device array instead of a caller workspace.

These tests call it through the C ABI, several calls in a row on the one shared
array, large calls before small ones, so a later call finds an earlier call's
bytes past its own region.  Each call's output must equal, bit for bit, what
the workspace-taking qlin_w8a8_linear computes on the same inputs (the same
kernels run), and must match the oracle within the layer's tolerance.  The
shapes reach every W8A8 kernel path: the INT8 in-GEMM quantization (M <= 64),
the INT8 separate pass, the E4M3 separate pass and the E4M3 cooperative GEMM
that quantizes inside itself and zeroes its task flags in the scratch.  Sizes
beyond the scratch are refused before any launch.

This file is named to be collected last.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from bit_quantized_linear_gb300 import synth
from _helpers import check_tol, from_dev_bf16, sample_rows

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
QT = {"int8": oracle.INT8, "e4m3": oracle.E4M3}

# call orders: the largest call first, so the smaller ones after it run over
# bytes it left in the scratch
ORDERS = {
    "int8": [(300, 2048, 272, "k_quantize_act_i8bf16+k_w8_dq<128,i8>"),
             (40, 1024, 384, "k_w8_dq<64,i8,xq>"),
             (7, 2048, 512, "k_w8_dq<16,i8,xq>")],
    "e4m3": [(8192, 4096, 2048, "k_fp8_gemm<xq>"),
             (300, 2048, 272, "k_quantize_act+k_fp8_gemm"),
             (77, 1024, 384, "k_quantize_act+k_fp8_gemm")],
}


@pytest.fixture(scope="module")
def capi():
    from bit_quantized_linear_gb300 import capi as c
    return c


def _case(qt, M, K, N, tag):
    rng = synth.rng_for("test-noalloc", 0, f"{qt}-{M}x{K}x{N}-{tag}", "all")
    outl = synth.outlier_channels(K, rng)
    w = synth.weights(N, K, rng)
    cal = synth.activations(1024, K, rng, outl)
    x = synth.activations(M, K, rng, outl)
    b = synth.bias(N, rng)
    q, s = oracle.quantize_weight(QT[qt], w)
    sx = oracle.act_scale(QT[qt], cal)
    return x, sx, q, s, b


def _dev(a, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else np.ascontiguousarray(a)).cuda()
    return t.view(torch.bfloat16) if bf16 else t


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_noalloc_equals_workspace_entry_point_in_a_row(capi, qt):
    for i, (M, K, N, kernel) in enumerate(ORDERS[qt]):
        assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, qt, M, K, N) == kernel
        assert capi.qlin_workspace_bytes(capi.QLIN_OP_W8A8_LINEAR, qt, M, K, N) <= capi.W8A8_NOALLOC_SCRATCH_BYTES
        x, sx, q, s, b = _case(qt, M, K, N, i)
        xd, qd, sd, bd = _dev(x, True), _dev(q), _dev(s), _dev(b, True)
        sxd = _dev(np.array([sx], np.float32))
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        capi.qlin_w8a8_linear_noalloc(qt, xd, sxd, qd, sd, bd, y)
        y_ws = capi.w8a8_linear(qt, xd, sxd, qd, sd, bd)
        torch.cuda.synchronize()
        assert capi.qlin_get_device_status() == capi.QLIN_OK
        assert torch.equal(y.view(torch.int16), y_ws.view(torch.int16)), f"noalloc {qt} call {i} {M}x{K}x{N}"
        rows = sample_rows(M, 24)
        ref = oracle.w8a8(QT[qt], oracle.quantize_act(QT[qt], x[rows], sx), sx, q, s, b)
        check_tol(from_dev_bf16(y)[rows], ref, f"noalloc {qt} call {i} {M}x{K}x{N} vs oracle")


def test_noalloc_repeats_bitwise(capi):
    """The same call twice in a row gives the same bits (the second finds the
    first one's codes and flags in the scratch)."""
    M, K, N = 8192, 4096, 2048
    x, sx, q, s, b = _case("e4m3", M, K, N, "repeat")
    xd, qd, sd, bd = _dev(x, True), _dev(q), _dev(s), _dev(b, True)
    sxd = _dev(np.array([sx], np.float32))
    y1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty_like(y1)
    capi.qlin_w8a8_linear_noalloc("e4m3", xd, sxd, qd, sd, bd, y1)
    capi.qlin_w8a8_linear_noalloc("e4m3", xd, sxd, qd, sd, bd, y2)
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_noalloc_rejects_sizes_beyond_scratch(capi):
    """The largest M whose workspace fits the scratch is accepted by the size
    check; one row more is refused with QLIN_ERR_WORKSPACE before any launch."""
    L = capi.lib()
    limit = capi.W8A8_NOALLOC_SCRATCH_BYTES
    src = open(os.path.join(ROOT, "include", "qlin.h")).read()
    assert re.search(r"QLIN_W8A8_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)64 << 20\)", src)
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
