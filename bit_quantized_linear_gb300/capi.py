"""Thin Python binding of libqlin (include/qlin.h): argument marshalling only.

Each ``qlin_*`` function takes torch tensors (device tensors for the data,
caller-allocated outputs), passes their device pointers, sizes and the current
CUDA stream to the C entry point of the same name, and raises QlinError on a
non-OK status.  No computation happens here; if the shared library is missing
the import fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqlin.so")

QLIN_OK, QLIN_ERR_INVALID_ARG, QLIN_ERR_UNSUPPORTED, QLIN_ERR_WORKSPACE, QLIN_ERR_CUDA, QLIN_ERR_TIMEOUT = range(6)
QLIN_INT8, QLIN_E4M3 = 0, 1
(QLIN_OP_QUANTIZE_WEIGHT, QLIN_OP_ACT_SCALE, QLIN_OP_QUANTIZE_ACT, QLIN_OP_W8A16_LINEAR,
 QLIN_OP_W8A8_LINEAR, QLIN_OP_I8_GEMM_S32, QLIN_OP_W8A8_DYNAMIC_LINEAR, QLIN_OP_KV_STORE_MIXED,
 QLIN_OP_KV_LOAD_MIXED, QLIN_OP_W8A16_GATE_UP_SILU, QLIN_OP_W8A8_GATE_UP_SILU) = range(11)

QTYPES = {"int8": QLIN_INT8, "e4m3": QLIN_E4M3}

# Every symbol the header declares (checked by the not-gpu ABI test).
EXPORTS = ["qlin_quantize_weight", "qlin_act_scale_from_calib", "qlin_quantize_act_static",
           "qlin_w8a16_linear", "qlin_w8a8_linear", "qlin_i8_gemm_s32", "qlin_workspace_bytes",
           "qlin_get_device_status", "qlin_status_string", "qlin_version", "qlin_debug_wait_flag",
           "qlin_kernel_name", "qlin_launch_count", "qlin_w8a8_linear_noalloc",
           "qlin_quantize_act_dynamic", "qlin_w8a8_dynamic_linear", "qlin_kv_store_mixed",
           "qlin_kv_load_mixed", "qlin_w8a16_gate_up_silu", "qlin_w8a8_gate_up_silu"]

# Size of the library-owned scratch of qlin_w8a8_linear_noalloc (QLIN_W8A8_NOALLOC_SCRATCH_BYTES).
W8A8_NOALLOC_SCRATCH_BYTES = 64 << 20


class QlinError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libqlin.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sig = {
        "qlin_quantize_weight": [I, I64, I64, P, P, P, P],
        "qlin_act_scale_from_calib": [I, I64, I64, P, P, P, SZ, P],
        "qlin_quantize_act_static": [I, I64, I64, P, P, P, P],
        "qlin_w8a16_linear": [I, I64, I64, I64, P, P, P, P, P, P, SZ, P],
        "qlin_w8a8_linear": [I, I64, I64, I64, P, P, P, P, P, P, P, SZ, P],
        "qlin_i8_gemm_s32": [I64, I64, I64, P, P, P, P, SZ, P],
        "qlin_workspace_bytes": [I, I, I64, I64, I64],
        "qlin_get_device_status": [P],
        "qlin_status_string": [I],
        "qlin_version": [],
        "qlin_debug_wait_flag": [P, ctypes.c_uint64, P],
        "qlin_kernel_name": [I, I, I64, I64, I64],
        "qlin_launch_count": [],
        "qlin_w8a8_linear_noalloc": [I, I64, I64, I64, P, P, P, P, P, P, P],
        "qlin_quantize_act_dynamic": [I, I64, I64, P, P, P, P],
        "qlin_w8a8_dynamic_linear": [I, I64, I64, I64, P, P, P, P, P, P, SZ, P],
        "qlin_kv_store_mixed": [I64, I64, I64, P, I64, P, I64, P, I64, P, P, P, P, P],
        "qlin_kv_load_mixed": [I64, I64, I64, P, I64, P, P, P, P, P, P, P],
        "qlin_w8a16_gate_up_silu": [I, I64, I64, I64, P, P, P, P, P, P, SZ, P],
        "qlin_w8a8_gate_up_silu": [I, I64, I64, I64, P, P, P, P, P, P, P, SZ, P],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = I
    L.qlin_workspace_bytes.restype = SZ
    L.qlin_status_string.restype = ctypes.c_char_p
    L.qlin_kernel_name.restype = ctypes.c_char_p
    L.qlin_launch_count.restype = ctypes.c_uint64
    return L


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def status_string(s: int) -> str:
    return _lib.qlin_status_string(int(s)).decode()


def _check(status: int, where: str):
    if status != QLIN_OK:
        raise QlinError(status, where)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _qt(qtype):
    return QTYPES[qtype] if isinstance(qtype, str) else int(qtype)


def qlin_workspace_bytes(op: int, qtype, M: int, K: int, N: int) -> int:
    return int(_lib.qlin_workspace_bytes(op, _qt(qtype), M, K, N))


def qlin_quantize_weight(qtype, w, qw, w_scale, stream=None):
    N, K = w.shape
    _check(_lib.qlin_quantize_weight(_qt(qtype), N, K, _p(w), _p(qw), _p(w_scale), _stream(stream)),
           "qlin_quantize_weight")


def qlin_act_scale_from_calib(qtype, x_cal, input_scale, ws, stream=None):
    rows, K = x_cal.shape
    _check(_lib.qlin_act_scale_from_calib(_qt(qtype), rows, K, _p(x_cal), _p(input_scale), _p(ws),
                                          0 if ws is None else ws.numel() * ws.element_size(),
                                          _stream(stream)), "qlin_act_scale_from_calib")


def qlin_quantize_act_static(qtype, x, input_scale, qx, stream=None):
    M, K = x.shape
    _check(_lib.qlin_quantize_act_static(_qt(qtype), M, K, _p(x), _p(input_scale), _p(qx), _stream(stream)),
           "qlin_quantize_act_static")


def _ws(ws):
    return (None, 0) if ws is None else (_p(ws), ws.numel() * ws.element_size())


def qlin_w8a16_linear(qtype, x, qw, w_scale, bias, y, ws=None, stream=None):
    M, K = x.shape
    N = qw.shape[0]
    wp, wb = _ws(ws)
    _check(_lib.qlin_w8a16_linear(_qt(qtype), M, K, N, _p(x), _p(qw), _p(w_scale), _p(bias), _p(y),
                                  wp, wb, _stream(stream)), "qlin_w8a16_linear")


def qlin_w8a8_linear(qtype, x, input_scale, qw, w_scale, bias, y, ws, stream=None):
    M, K = x.shape
    N = qw.shape[0]
    wp, wb = _ws(ws)
    _check(_lib.qlin_w8a8_linear(_qt(qtype), M, K, N, _p(x), _p(input_scale), _p(qw), _p(w_scale),
                                 _p(bias), _p(y), wp, wb, _stream(stream)), "qlin_w8a8_linear")


def qlin_w8a8_linear_noalloc(qtype, x, input_scale, qw, w_scale, bias, y, stream=None):
    """W8A8 static linear without a workspace (see qlin_w8a8_linear_noalloc in
    include/qlin.h): for callers that cannot allocate device memory."""
    M, K = x.shape
    N = qw.shape[0]
    _check(_lib.qlin_w8a8_linear_noalloc(_qt(qtype), M, K, N, _p(x), _p(input_scale), _p(qw), _p(w_scale),
                                         _p(bias), _p(y), _stream(stream)), "qlin_w8a8_linear_noalloc")


def qlin_quantize_act_dynamic(qtype, x, qx, x_scale, stream=None):
    M, K = x.shape
    _check(_lib.qlin_quantize_act_dynamic(_qt(qtype), M, K, _p(x), _p(qx), _p(x_scale), _stream(stream)),
           "qlin_quantize_act_dynamic")


def qlin_w8a8_dynamic_linear(qtype, x, qw, w_scale, bias, y, ws, stream=None):
    M, K = x.shape
    N = qw.shape[0]
    wp, wb = _ws(ws)
    _check(_lib.qlin_w8a8_dynamic_linear(_qt(qtype), M, K, N, _p(x), _p(qw), _p(w_scale), _p(bias), _p(y),
                                         wp, wb, _stream(stream)), "qlin_w8a8_dynamic_linear")


def qlin_i8_gemm_s32(qx, qw, acc, ws=None, stream=None):
    M, K = qx.shape
    N = qw.shape[0]
    wp, wb = _ws(ws)
    _check(_lib.qlin_i8_gemm_s32(M, K, N, _p(qx), _p(qw), _p(acc), wp, wb, _stream(stream)),
           "qlin_i8_gemm_s32")


def qlin_w8a16_gate_up_silu(qtype, x, qw, w_scale, bias, y, ws=None, stream=None):
    """qw [2I, K] (gate rows first), y [M, I]."""
    M, K = x.shape
    I = qw.shape[0] // 2
    wp, wb = _ws(ws)
    _check(_lib.qlin_w8a16_gate_up_silu(_qt(qtype), M, K, I, _p(x), _p(qw), _p(w_scale), _p(bias), _p(y), wp, wb,
                                        _stream(stream)), "qlin_w8a16_gate_up_silu")


def qlin_w8a8_gate_up_silu(qtype, x, input_scale, qw, w_scale, bias, y, ws, stream=None):
    M, K = x.shape
    I = qw.shape[0] // 2
    wp, wb = _ws(ws)
    _check(_lib.qlin_w8a8_gate_up_silu(_qt(qtype), M, K, I, _p(x), _p(input_scale), _p(qw), _p(w_scale), _p(bias),
                                       _p(y), wp, wb, _stream(stream)), "qlin_w8a8_gate_up_silu")


def qlin_kv_store_mixed(k, v, slots, k_cache, k_scale, v_cache, v_scale, stream=None):
    """k, v: BF16 [T, ld] (row stride ld elements, last dim contiguous); slots int64 [T];
    caches as allocated by kv_cache_alloc()."""
    S, H, D = k_cache.shape
    T = slots.shape[0]
    assert k.stride(-1) == 1 and v.stride(-1) == 1
    ldk = k.stride(0) if T > 0 else H * D
    ldv = v.stride(0) if T > 0 else H * D
    _check(_lib.qlin_kv_store_mixed(T, H, D, _p(k), ldk, _p(v), ldv, _p(slots), S, _p(k_cache), _p(k_scale),
                                    _p(v_cache), _p(v_scale), _stream(stream)), "qlin_kv_store_mixed")


def qlin_kv_load_mixed(slots, k_cache, k_scale, v_cache, v_scale, k_out, v_out, stream=None):
    S, H, D = k_cache.shape
    T = slots.shape[0]
    _check(_lib.qlin_kv_load_mixed(T, H, D, _p(slots), S, _p(k_cache), _p(k_scale), _p(v_cache), _p(v_scale),
                                   _p(k_out), _p(v_out), _stream(stream)), "qlin_kv_load_mixed")


def qlin_kernel_name(op: int, qtype, M: int, K: int, N: int) -> str:
    return _lib.qlin_kernel_name(op, _qt(qtype), M, K, N).decode()


def qlin_launch_count() -> int:
    return int(_lib.qlin_launch_count())


def qlin_get_device_status(stream=None) -> int:
    return int(_lib.qlin_get_device_status(_stream(stream)))


def qlin_debug_wait_flag(flag, timeout_ns: int, stream=None):
    _check(_lib.qlin_debug_wait_flag(_p(flag), int(timeout_ns), _stream(stream)), "qlin_debug_wait_flag")


# ---------------------------------------------------------------------------
# Convenience wrappers that allocate outputs / workspaces with torch (device
# memory only) and call the entry points above.
# ---------------------------------------------------------------------------
def workspace(op: int, qtype, M: int, K: int, N: int, device=None):
    n = qlin_workspace_bytes(op, qtype, M, K, N)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def quantize_weight(qtype, w):
    N, K = w.shape
    qw = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((N,), dtype=torch.float32, device=w.device)
    qlin_quantize_weight(qtype, w, qw, s)
    return qw, s


def act_scale_from_calib(qtype, x_cal):
    s = torch.empty((1,), dtype=torch.float32, device=x_cal.device)
    ws = workspace(QLIN_OP_ACT_SCALE, qtype, *x_cal.shape, 0, device=x_cal.device)
    qlin_act_scale_from_calib(qtype, x_cal, s, ws)
    return s


def quantize_act_static(qtype, x, input_scale):
    qx = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    qlin_quantize_act_static(qtype, x, input_scale, qx)
    return qx


def w8a16_linear(qtype, x, qw, w_scale, bias=None):
    M, K = x.shape
    N = qw.shape[0]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws = workspace(QLIN_OP_W8A16_LINEAR, qtype, M, K, N, device=x.device)
    qlin_w8a16_linear(qtype, x, qw, w_scale, bias, y, ws)
    return y


def w8a8_linear(qtype, x, input_scale, qw, w_scale, bias=None):
    M, K = x.shape
    N = qw.shape[0]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws = workspace(QLIN_OP_W8A8_LINEAR, qtype, M, K, N, device=x.device)
    qlin_w8a8_linear(qtype, x, input_scale, qw, w_scale, bias, y, ws)
    return y


def quantize_act_dynamic(qtype, x):
    qx = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    s = torch.empty((x.shape[0],), dtype=torch.float32, device=x.device)
    qlin_quantize_act_dynamic(qtype, x, qx, s)
    return qx, s


def w8a8_dynamic_linear(qtype, x, qw, w_scale, bias=None):
    M, K = x.shape
    N = qw.shape[0]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws = workspace(QLIN_OP_W8A8_DYNAMIC_LINEAR, qtype, M, K, N, device=x.device)
    qlin_w8a8_dynamic_linear(qtype, x, qw, w_scale, bias, y, ws)
    return y


def i8_gemm_s32(qx, qw):
    M, K = qx.shape
    N = qw.shape[0]
    acc = torch.empty((M, N), dtype=torch.int32, device=qx.device)
    ws = workspace(QLIN_OP_I8_GEMM_S32, QLIN_INT8, M, K, N, device=qx.device)
    qlin_i8_gemm_s32(qx, qw, acc, ws)
    return acc


def kv_cache_alloc(num_slots: int, H: int, D: int, device=None):
    """Device arrays of a mixed KV cache: k_cache int8 [S,H,D], k_scale float16 bits
    [S,H,D/32] (int16 storage), v_cache E4M3 codes [S,H,D] (uint8), v_scale float16
    bits [S,H] (int16 storage)."""
    dev = device or "cuda"
    return (torch.empty((num_slots, H, D), dtype=torch.int8, device=dev),
            torch.empty((num_slots, H, D // 32), dtype=torch.int16, device=dev),
            torch.empty((num_slots, H, D), dtype=torch.uint8, device=dev),
            torch.empty((num_slots, H), dtype=torch.int16, device=dev))


def kv_load_mixed(slots, cache):
    S, H, D = cache[0].shape
    T = slots.shape[0]
    k = torch.empty((T, H, D), dtype=torch.bfloat16, device=slots.device)
    v = torch.empty((T, H, D), dtype=torch.bfloat16, device=slots.device)
    qlin_kv_load_mixed(slots, *cache, k, v)
    return k, v


def w8a16_gate_up_silu(qtype, x, qw, w_scale, bias=None):
    M, K = x.shape
    I = qw.shape[0] // 2
    y = torch.empty((M, I), dtype=torch.bfloat16, device=x.device)
    ws = workspace(QLIN_OP_W8A16_GATE_UP_SILU, qtype, M, K, I, device=x.device)
    qlin_w8a16_gate_up_silu(qtype, x, qw, w_scale, bias, y, ws)
    return y


def w8a8_gate_up_silu(qtype, x, input_scale, qw, w_scale, bias=None):
    M, K = x.shape
    I = qw.shape[0] // 2
    y = torch.empty((M, I), dtype=torch.bfloat16, device=x.device)
    ws = workspace(QLIN_OP_W8A8_GATE_UP_SILU, qtype, M, K, I, device=x.device)
    qlin_w8a8_gate_up_silu(qtype, x, input_scale, qw, w_scale, bias, y, ws)
    return y
