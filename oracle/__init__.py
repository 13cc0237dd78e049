"""qlin oracle: TEST INFRASTRUCTURE ONLY.

A plain CPU restatement (C, fp64 / exact integer arithmetic) of the 8-bit
quantized linear layer: per-output-channel weight quantizers (INT8 and OCP
E4M3), the static activation scale from a calibration batch, static activation
quantization, the exact INT8 accumulator, the fp64 W8A8 / W8A16 references and
the mixed KV-cache quantizers (INT8 keys with float16 group scales, E4M3 values
with float16 per-token scales) and the merged gate_up linear with the SiLU * up
epilogue.
The C source ``qlin_oracle.c`` cites the passages it follows.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  It shares no code with the CUDA library; the product
path never loads it.  Every function is pinned by a not-gpu test.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qlin_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

INT8 = 0
E4M3 = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2 -fopenmp, no fast-math, no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_encode.argtypes = [ctypes.c_double]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_quantize_weight.argtypes = [I, I64, I64, P, P, P]
            L.orc_quantize_weight.restype = None
            L.orc_act_scale.argtypes = [I, I64, I64, P]
            L.orc_act_scale.restype = ctypes.c_float
            L.orc_quantize_act.argtypes = [I, I64, I64, P, ctypes.c_float, P]
            L.orc_quantize_act.restype = None
            L.orc_i8_gemm.argtypes = [I64, I64, I64, P, P, P]
            L.orc_i8_gemm.restype = I64
            L.orc_w8a8.argtypes = [I, I64, I64, I64, P, ctypes.c_float, P, P, P, P, I64, P]
            L.orc_w8a8.restype = None
            L.orc_w8a16.argtypes = [I, I64, I64, I64, P, P, P, P, P, I64, P]
            L.orc_w8a16.restype = None
            L.orc_quantize_act_per_token.argtypes = [I, I64, I64, P, P, P]
            L.orc_quantize_act_per_token.restype = None
            L.orc_w8a8_per_token.argtypes = [I, I64, I64, I64, P, P, P, P, P, P, I64, P]
            L.orc_w8a8_per_token.restype = None
            L.orc_fp16_decode.argtypes = [ctypes.c_uint16]
            L.orc_fp16_decode.restype = ctypes.c_double
            L.orc_fp16_encode.argtypes = [ctypes.c_double]
            L.orc_fp16_encode.restype = ctypes.c_uint16
            L.orc_bf16_encode.argtypes = [ctypes.c_double]
            L.orc_bf16_encode.restype = ctypes.c_uint16
            L.orc_kv_store.argtypes = [I64, I64, I64, P, I64, P, I64, P, I64, P, P, P, P]
            L.orc_kv_store.restype = I64
            L.orc_kv_load.argtypes = [I64, I64, I64, P, I64, P, P, P, P, P, P]
            L.orc_kv_load.restype = I64
            L.orc_w8a16_gate_up_silu.argtypes = [I, I64, I64, I64, P, P, P, P, P, I64, P]
            L.orc_w8a16_gate_up_silu.restype = I
            L.orc_w8a8_gate_up_silu.argtypes = [I, I64, I64, I64, P, ctypes.c_float, P, P, P, P, I64, P]
            L.orc_w8a8_gate_up_silu.restype = I
            L.orc_num_threads.argtypes = []
            L.orc_num_threads.restype = I
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def quantize_weight(qtype: int, w: np.ndarray):
    """w: float32 [N,K] -> (q uint8 [N,K] (int8 bits or E4M3 codes), s float32 [N])."""
    w = _c(w, np.float32)
    N, K = w.shape
    q = np.empty((N, K), np.uint8)
    s = np.empty((N,), np.float32)
    lib().orc_quantize_weight(qtype, N, K, _ptr(w), _ptr(q), _ptr(s))
    return q, s


def act_scale(qtype: int, x_cal_bf16: np.ndarray) -> np.float32:
    """x_cal: uint16 BF16 bits [rows,K] -> fp32 per-tensor input scale."""
    x = _c(x_cal_bf16, np.uint16)
    rows, K = x.shape
    return np.float32(lib().orc_act_scale(qtype, rows, K, _ptr(x)))


def quantize_act(qtype: int, x_bf16: np.ndarray, s_x) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    lib().orc_quantize_act(qtype, M, K, _ptr(x), ctypes.c_float(float(np.float32(s_x))), _ptr(q))
    return q


def i8_gemm(qx: np.ndarray, qw: np.ndarray) -> np.ndarray:
    """Exact int32 accumulator sum_k qx[m,k]*qw[n,k] (int8 inputs)."""
    qx = _c(qx.view(np.int8), np.int8)
    qw = _c(qw.view(np.int8), np.int8)
    M, K = qx.shape
    N, K2 = qw.shape
    assert K == K2
    acc = np.empty((M, N), np.int32)
    bad = lib().orc_i8_gemm(M, K, N, _ptr(qx), _ptr(qw), _ptr(acc))
    if bad:
        raise OverflowError(f"{bad} accumulator entries exceed int32")
    return acc


def _rows(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, np.int64))
    assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < M))
    return r, r.size


def w8a8(qtype: int, qx, s_x, qw, s_w, bias=None, rows=None) -> np.ndarray:
    """fp64 W8A8 reference y[rows or all, N]."""
    qx = _c(qx, np.uint8)
    qw = _c(qw, np.uint8)
    s_w = _c(s_w, np.float32)
    M, K = qx.shape
    N = qw.shape[0]
    b = None if bias is None else _c(bias, np.uint16)
    r, R = _rows(rows, M)
    y = np.empty((R, N), np.float64)
    lib().orc_w8a8(qtype, M, K, N, _ptr(qx), ctypes.c_float(float(np.float32(s_x))), _ptr(qw),
                   _ptr(s_w), _ptr(b), _ptr(r), R, _ptr(y))
    return y


def w8a16(qtype: int, x_bf16, qw, s_w, bias=None, rows=None) -> np.ndarray:
    """fp64 W8A16 reference y[rows or all, N]."""
    x = _c(x_bf16, np.uint16)
    qw = _c(qw, np.uint8)
    s_w = _c(s_w, np.float32)
    M, K = x.shape
    N = qw.shape[0]
    b = None if bias is None else _c(bias, np.uint16)
    r, R = _rows(rows, M)
    y = np.empty((R, N), np.float64)
    lib().orc_w8a16(qtype, M, K, N, _ptr(x), _ptr(qw), _ptr(s_w), _ptr(b), _ptr(r), R, _ptr(y))
    return y


def quantize_act_per_token(qtype: int, x_bf16):
    """Dynamic per-token quantization: (q uint8 [M,K], s_x float32 [M])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((M,), np.float32)
    lib().orc_quantize_act_per_token(qtype, M, K, _ptr(x), _ptr(s), _ptr(q))
    return q, s


def w8a8_per_token(qtype: int, qx, s_x, qw, s_w, bias=None, rows=None) -> np.ndarray:
    """fp64 W8A8 reference with one activation scale per token row."""
    qx = _c(qx, np.uint8)
    qw = _c(qw, np.uint8)
    s_x = _c(s_x, np.float32)
    s_w = _c(s_w, np.float32)
    M, K = qx.shape
    N = qw.shape[0]
    b = None if bias is None else _c(bias, np.uint16)
    r, R = _rows(rows, M)
    y = np.empty((R, N), np.float64)
    lib().orc_w8a8_per_token(qtype, M, K, N, _ptr(qx), _ptr(s_x), _ptr(qw), _ptr(s_w), _ptr(b), _ptr(r), R,
                             _ptr(y))
    return y


def w8a16_gate_up_silu(qtype: int, x_bf16, qw, s_w, bias=None, rows=None) -> np.ndarray:
    """fp64 silu(gate) * up of a merged gate_up W8A16 linear: qw [2I, K] (gate rows
    first), s_w [2I], bias [2I] or None -> y [rows or M, I]."""
    x = _c(x_bf16, np.uint16)
    qw = _c(qw, np.uint8)
    s_w = _c(s_w, np.float32)
    M, K = x.shape
    assert qw.shape[0] % 2 == 0
    I = qw.shape[0] // 2
    b = None if bias is None else _c(bias, np.uint16)
    r, R = _rows(rows, M)
    y = np.empty((R, I), np.float64)
    if lib().orc_w8a16_gate_up_silu(qtype, M, K, I, _ptr(x), _ptr(qw), _ptr(s_w), _ptr(b), _ptr(r), R, _ptr(y)):
        raise MemoryError("oracle temporary")
    return y


def w8a8_gate_up_silu(qtype: int, qx, s_x, qw, s_w, bias=None, rows=None) -> np.ndarray:
    """fp64 silu(gate) * up of a merged gate_up W8A8 static linear."""
    qx = _c(qx, np.uint8)
    qw = _c(qw, np.uint8)
    s_w = _c(s_w, np.float32)
    M, K = qx.shape
    I = qw.shape[0] // 2
    b = None if bias is None else _c(bias, np.uint16)
    r, R = _rows(rows, M)
    y = np.empty((R, I), np.float64)
    if lib().orc_w8a8_gate_up_silu(qtype, M, K, I, _ptr(qx), ctypes.c_float(float(np.float32(s_x))), _ptr(qw),
                                   _ptr(s_w), _ptr(b), _ptr(r), R, _ptr(y)):
        raise MemoryError("oracle temporary")
    return y


def fp16_decode(code: int) -> float:
    return lib().orc_fp16_decode(int(code) & 0xFFFF)


def fp16_encode(v: float) -> int:
    return int(lib().orc_fp16_encode(float(v)))


def bf16_encode(v: float) -> int:
    return int(lib().orc_bf16_encode(float(v)))


class KVCache:
    """Host copy of a mixed KV cache with num_slots slots, H kv heads and head
    size D: k_cache int8 bits [S,H,D], k_scale float16 bits [S,H,D/32], v_cache
    E4M3 codes [S,H,D], v_scale float16 bits [S,H].  Every byte starts as `fill`."""

    def __init__(self, num_slots: int, H: int, D: int, fill: int = 0):
        assert D % 32 == 0
        self.num_slots, self.H, self.D = num_slots, H, D
        self.k_cache = np.full((num_slots, H, D), fill & 0xFF, np.uint8)
        self.k_scale = np.full((num_slots, H, D // 32), (fill & 0xFF) * 0x0101, np.uint16)
        self.v_cache = np.full((num_slots, H, D), fill & 0xFF, np.uint8)
        self.v_scale = np.full((num_slots, H), (fill & 0xFF) * 0x0101, np.uint16)

    def nbytes(self) -> int:
        return sum(a.nbytes for a in (self.k_cache, self.k_scale, self.v_cache, self.v_scale))


def kv_store(cache: KVCache, k_bf16, v_bf16, slots) -> int:
    """Quantizes token rows k, v (uint16 BF16 bits [T, ld >= H*D]) into cache
    slots; negative slots are skipped.  Returns the count of slots >= num_slots."""
    k = _c(k_bf16, np.uint16)
    v = _c(v_bf16, np.uint16)
    sl = _c(np.asarray(slots, np.int64), np.int64)
    T = sl.shape[0]
    H, D = cache.H, cache.D
    assert k.shape[0] == T and v.shape[0] == T and k.shape[1] >= H * D and v.shape[1] >= H * D
    return int(lib().orc_kv_store(T, H, D, _ptr(k), k.shape[1], _ptr(v), v.shape[1], _ptr(sl), cache.num_slots,
                                  _ptr(cache.k_cache), _ptr(cache.k_scale), _ptr(cache.v_cache),
                                  _ptr(cache.v_scale)))


def kv_load(cache: KVCache, slots):
    """Dequantizes cache slots to BF16 bits (k_out, v_out) [T,H,D] and the count
    of slots >= num_slots; negative or out-of-range slots give rows of +0."""
    sl = _c(np.asarray(slots, np.int64), np.int64)
    T = sl.shape[0]
    H, D = cache.H, cache.D
    ko = np.empty((T, H, D), np.uint16)
    vo = np.empty((T, H, D), np.uint16)
    bad = lib().orc_kv_load(T, H, D, _ptr(sl), cache.num_slots, _ptr(cache.k_cache), _ptr(cache.k_scale),
                            _ptr(cache.v_cache), _ptr(cache.v_scale), _ptr(ko), _ptr(vo))
    return ko, vo, int(bad)


def num_threads() -> int:
    return int(lib().orc_num_threads())
