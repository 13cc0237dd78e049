"""Host-side checks of the C ABI (not gpu): the library loads, exports every
function include/qlin.h declares, and rejects bad arguments before touching a
device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def capi():
    from bit_quantized_linear_gb300 import build
    build.build()
    from bit_quantized_linear_gb300 import capi as c
    return c


def declared_functions():
    src = open(os.path.join(ROOT, "include", "qlin.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qlin_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["qlin_quantize_weight", "qlin_quantize_act_static", "qlin_w8a16_linear", "qlin_w8a8_linear",
              "qlin_act_scale_from_calib", "qlin_i8_gemm_s32", "qlin_workspace_bytes"]:
        assert n in names


def test_library_exports_every_declared_symbol(capi):
    L = ctypes.CDLL(capi.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    assert sorted(capi.EXPORTS) == declared_functions()


def test_status_strings_and_version(capi):
    assert capi.status_string(0) == "QLIN_OK"
    assert capi.status_string(5) == "QLIN_ERR_TIMEOUT"
    assert capi.lib().qlin_version() >= 100


def test_workspace_sizes(capi):
    ws = capi.qlin_workspace_bytes
    assert ws(capi.QLIN_OP_ACT_SCALE, "int8", 32768, 2048, 0) >= 4
    assert ws(capi.QLIN_OP_W8A8_LINEAR, "e4m3", 1024, 2048, 11008) >= 1024 * 2048
    assert ws(capi.QLIN_OP_W8A8_LINEAR, "int8", 0, 2048, 11008) == 0
    assert ws(capi.QLIN_OP_W8A16_LINEAR, 7, 1, 16, 16) == 2 ** 64 - 1


def test_invalid_arguments_rejected_on_host(capi):
    L = capi.lib()
    P = ctypes.c_void_p
    good = P(4096)  # never dereferenced: validation fails before any launch
    odd = P(4096 + 8)
    INV, WS = capi.QLIN_ERR_INVALID_ARG, capi.QLIN_ERR_WORKSPACE
    # unknown qtype
    assert L.qlin_w8a16_linear(9, 1, 64, 64, good, good, good, None, good, None, 0, None) == INV
    # K, N not multiples of 16 / too small / negative M
    assert L.qlin_w8a16_linear(0, 1, 72, 64, good, good, good, None, good, None, 0, None) == INV
    assert L.qlin_w8a16_linear(0, 1, 64, 40, good, good, good, None, good, None, 0, None) == INV
    assert L.qlin_w8a16_linear(0, -1, 64, 64, good, good, good, None, good, None, 0, None) == INV
    assert L.qlin_w8a16_linear(0, 1, 0, 64, good, good, good, None, good, None, 0, None) == INV
    # NULL and misaligned pointers
    assert L.qlin_w8a16_linear(0, 1, 64, 64, None, good, good, None, good, None, 0, None) == INV
    assert L.qlin_w8a16_linear(0, 1, 64, 64, odd, good, good, None, good, None, 0, None) == INV
    assert L.qlin_w8a16_linear(0, 1, 64, 64, good, good, good, odd, good, None, 0, None) == INV
    # W8A8 needs a workspace large enough for the quantized activations
    assert L.qlin_w8a8_linear(1, 4, 64, 64, good, good, good, good, None, good, None, 0, None) == WS
    assert L.qlin_w8a8_linear(1, 4, 64, 64, good, good, good, good, None, good, good, 16, None) == WS
    assert L.qlin_act_scale_from_calib(0, 8, 64, good, good, None, 0, None) == WS
    assert L.qlin_quantize_weight(0, 4, 24, good, good, good, None) == INV
    assert L.qlin_quantize_act_static(1, 4, 64, good, None, good, None) == INV
    assert L.qlin_i8_gemm_s32(4, 64, 64, good, good, None, None, 0, None) == INV
    assert L.qlin_i8_gemm_s32(4, 64, 64, good, None, good, None, 0, None) == INV
    assert L.qlin_debug_wait_flag(None, 1000, None) == INV
    # KV cache: head_dim outside {32,64,128,256}, bad strides, NULL / misaligned pointers
    kv_store = lambda T, H, D, k, ldk, ldv, sl, kc: L.qlin_kv_store_mixed(T, H, D, k, ldk, good, ldv, sl, 64, kc,
                                                                          good, good, good, None)
    assert kv_store(4, 2, 96, good, 192, 192, good, good) == INV
    assert kv_store(4, 2, 128, good, 200, 256, good, good) == INV  # ldk not a multiple of 8
    assert kv_store(4, 2, 128, good, 248, 256, good, good) == INV  # ldk < H*D
    assert kv_store(4, 2, 128, None, 256, 256, good, good) == INV
    assert kv_store(4, 2, 128, odd, 256, 256, good, good) == INV
    assert kv_store(4, 2, 128, good, 256, 256, None, good) == INV
    assert kv_store(4, 0, 128, good, 256, 256, good, good) == INV
    assert kv_store(-1, 2, 128, good, 256, 256, good, good) == INV
    assert L.qlin_kv_load_mixed(4, 2, 128, good, 64, good, good, good, good, None, good, None) == INV
    assert L.qlin_kv_load_mixed(4, 2, 128, good, 64, good, odd, good, good, good, good, None) == INV
    assert L.qlin_kv_load_mixed(4, 2, 48, good, 64, good, good, good, good, good, good, None) == INV
    assert capi.qlin_kernel_name(capi.QLIN_OP_KV_STORE_MIXED, 0, 8, 128, 4) == "k_kv_store_mixed<128>"
    assert capi.qlin_kernel_name(capi.QLIN_OP_KV_LOAD_MIXED, 0, 8, 64, 4) == "k_kv_load_mixed<64>"
    assert capi.qlin_kernel_name(capi.QLIN_OP_KV_LOAD_MIXED, 0, 8, 80, 4) == "invalid"
    # merged gate_up: I a multiple of 128; W8A8 needs its workspace
    assert L.qlin_w8a16_gate_up_silu(0, 4, 64, 192, good, good, good, None, good, None, 0, None) == INV
    assert L.qlin_w8a16_gate_up_silu(0, 4, 64, 0, good, good, good, None, good, None, 0, None) == INV
    assert L.qlin_w8a16_gate_up_silu(0, 4, 64, 128, odd, good, good, None, good, None, 0, None) == INV
    assert L.qlin_w8a8_gate_up_silu(1, 4, 64, 128, good, good, good, good, None, good, None, 0, None) == WS
    assert L.qlin_w8a8_gate_up_silu(1, 4, 64, 100, good, good, good, good, None, good, good, 4096, None) == INV
    assert capi.qlin_workspace_bytes(capi.QLIN_OP_W8A8_GATE_UP_SILU, "e4m3", 4, 64, 128) >= 256
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A16_GATE_UP_SILU, 0, 1, 3584, 18944) == "k_w8_dq<16>"
    # E4M3 weights up to 128 tokens: FP8 MMAs against the split activations; above, the BF16 path
    for m, name in [(1, "k_w8a16_split+k_w8a16_f8<16>"), (16, "k_w8a16_split+k_w8a16_f8<16>"),
                    (17, "k_w8a16_split+k_w8a16_f8<32>"), (32, "k_w8a16_split+k_w8a16_f8<32>"),
                    (33, "k_w8_dq<64>")]:
        assert capi.qlin_kernel_name(capi.QLIN_OP_W8A16_LINEAR, 1, m, 3584, 3584) == name, m
    assert capi.qlin_workspace_bytes(capi.QLIN_OP_W8A16_LINEAR, "e4m3", 1, 3584, 3584) > 0
    assert capi.qlin_workspace_bytes(capi.QLIN_OP_W8A16_LINEAR, "int8", 1, 3584, 3584) == 0
    assert capi.qlin_workspace_bytes(capi.QLIN_OP_W8A16_LINEAR, "e4m3", 33, 3584, 3584) == 0
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_GATE_UP_SILU, 1, 8192, 2048, 11008) == "k_quantize_act+k_fp8_gemm"
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_GATE_UP_SILU, 1, 8192, 4096, 1024) == "k_fp8_gemm<xq>"
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, 1, 8192, 11008, 2048) == "k_fp8_gemm<xq>"
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, 1, 8192, 4096, 4096) == "k_fp8_gemm<xq>"
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, 1, 8192, 4096, 4112) == "k_quantize_act+k_fp8_gemm"
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, 1, 8192, 2048, 2048) == "k_quantize_act+k_fp8_gemm"
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, 1, 8064, 11008, 2048) == "k_quantize_act+k_fp8_gemm"
    # one n-tile: the tiles would not fill the SMs
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, 1, 8192, 11008, 256) == "k_quantize_act+k_fp8_gemm"
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, 1, 1024, 2048, 11008) == "k_quantize_act+k_fp8_gemm"


def test_no_device_is_reported_not_crashed(capi):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    L = capi.lib()
    P = ctypes.c_void_p
    good = P(4096)
    st = L.qlin_w8a16_linear(0, 1, 64, 64, good, good, good, None, good, None, 0, None)
    assert st in (capi.QLIN_ERR_UNSUPPORTED, capi.QLIN_ERR_CUDA)


def test_fused_quant_switch_selects_the_separate_pass():
    """QLIN_FP8_FUSED_QUANT=0 (read once per process) routes E4M3 W8A8 through
    the separate quantization pass, for every size."""
    import subprocess
    import sys
    code = ("from bit_quantized_linear_gb300 import capi; "
            "print(capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, 1, 8192, 11008, 2048)); "
            "print(capi.qlin_kernel_name(capi.QLIN_OP_W8A8_GATE_UP_SILU, 1, 8192, 4096, 1024))")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, QLIN_FP8_FUSED_QUANT="0", PYTHONPATH=root)
    out = subprocess.run([sys.executable, "-c", code], env=env, cwd=root, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.split() == ["k_quantize_act+k_fp8_gemm"] * 2
    env["QLIN_FP8_FUSED_QUANT"] = "1"
    out = subprocess.run([sys.executable, "-c", code], env=env, cwd=root, capture_output=True, text=True,
                         timeout=300)
    assert out.stdout.split() == ["k_fp8_gemm<xq>"] * 2


def test_noalloc_reports_as_the_workspace_entry_point(capi):
    """qlin_w8a8_linear_noalloc makes qlin_w8a8_linear's checks in the same
    order (arguments, size, device), so both return the same status for the
    same bad call.  Calls that pass every argument check reach the device check
    only where no device is present (they would launch on fake pointers)."""
    import torch
    L = capi.lib()
    P = ctypes.c_void_p
    good, odd = P(4096), P(4096 + 8)
    big_ws = 1 << 40  # never dereferenced: every call below stops before a launch

    def both(qt, M, K, N, x, sx, qw, s, b, y):
        ws = L.qlin_w8a8_linear(qt, M, K, N, x, sx, qw, s, b, y, good, big_ws, None)
        na = L.qlin_w8a8_linear_noalloc(qt, M, K, N, x, sx, qw, s, b, y, None)
        return ws, na

    INV = capi.QLIN_ERR_INVALID_ARG
    bad = [(9, 4, 64, 64, good, good, good, good, None, good),     # unknown qtype
           (0, 4, 72, 64, good, good, good, good, None, good),     # K not a multiple of 16
           (1, 4, 64, 40, good, good, good, good, None, good),     # N not a multiple of 16
           (1, -1, 64, 64, good, good, good, good, None, good),    # negative M
           (0, 4, 64, 64, None, good, good, good, None, good),     # no x
           (1, 4, 64, 64, good, None, good, good, None, good),     # no input_scale
           (1, 4, 64, 64, good, P(4098), good, good, None, good),  # input_scale not 4-byte aligned
           (0, 4, 64, 64, good, good, odd, good, None, good),      # qw misaligned
           (1, 4, 64, 64, good, good, good, good, odd, good),      # bias misaligned
           (0, 4, 64, 64, good, good, good, good, None, odd)]      # y misaligned
    for args in bad:
        assert both(*args) == (INV, INV), args
    # beyond the scratch: the size check answers before the device check
    assert L.qlin_w8a8_linear_noalloc(1, 65536, 2048, 64, good, good, good, good, None, good, None) == \
        capi.QLIN_ERR_WORKSPACE
    assert L.qlin_w8a8_linear(1, 65536, 2048, 64, good, good, good, good, None, good, good, 64 << 20, None) == \
        capi.QLIN_ERR_WORKSPACE
    if not torch.cuda.is_available():
        for args in [(1, 0, 64, 64, None, good, good, good, None, None), (0, 4, 64, 64, good, good, good, good, None, good)]:
            ws, na = both(*args)
            assert ws == na and ws in (capi.QLIN_ERR_UNSUPPORTED, capi.QLIN_ERR_CUDA), (args, ws, na)


def test_fp8_w8a16_token_tiles(capi):
    """E4M3 W8A16 up to 32 tokens: the split activations take 4 x tt rows of K
    bytes per token tile of tt tokens (tt = 4, 8, 16 or 32, the least that holds
    the batch up to 16 tokens), each region rounded up to 256 bytes, and one fp32
    scale per token."""
    K = 3584
    up = lambda b: (b + 255) // 256 * 256
    for m, tt in [(1, 4), (4, 4), (5, 8), (8, 8), (9, 16), (16, 16), (17, 32), (32, 32)]:
        tiles = (m + tt - 1) // tt
        want = up(tiles * 4 * tt * K) + up(4 * m)
        assert capi.qlin_workspace_bytes(capi.QLIN_OP_W8A16_LINEAR, "e4m3", m, K, 4096) == want, m
        kernel = "k_w8a16_split+k_w8a16_f8<16>" if m <= 16 else "k_w8a16_split+k_w8a16_f8<32>"
        assert capi.qlin_kernel_name(capi.QLIN_OP_W8A16_LINEAR, "e4m3", m, K, 4096) == kernel, m
