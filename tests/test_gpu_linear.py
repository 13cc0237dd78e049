"""GPU parity of the linears against the oracle (through the C ABI).

BF16 outputs: within the stated tolerance of the fp64 oracle on the SAME
quantized operands (so only accumulation and output rounding are measured).
INT8 accumulator: bit-exact.  Full-size workloads are checked on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_quantized_linear_gb300 import synth
from _helpers import check_tol, from_dev_bf16, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
QT = {"int8": oracle.INT8, "e4m3": oracle.E4M3}


@pytest.fixture(scope="module")
def capi():
    from bit_quantized_linear_gb300 import capi as c
    return c


def _operands(lin, rows=None):
    t = synth.make_inputs(lin)
    q, s = oracle.quantize_weight(QT[lin.qtype], t["w"])
    return t, q, s


def run_w8a16(capi, qt, x, q, s, b):
    y = capi.w8a16_linear(qt, to_dev_bf16(x), to_dev(q), to_dev(s), None if b is None else to_dev_bf16(b))
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    return from_dev_bf16(y)


def run_w8a8(capi, qt, x, sx, q, s, b):
    y = capi.w8a8_linear(qt, to_dev_bf16(x), to_dev(np.array([sx], np.float32)), to_dev(q), to_dev(s),
                         None if b is None else to_dev_bf16(b))
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    return from_dev_bf16(y)


# ----------------------------------------------------------------- W8A16
def w8a16_case(capi, qt, M, K, N, with_bias, seed_tag, rows=None, outliers=False):
    rng = synth.rng_for("test-w8a16", 0, f"{qt}-{M}x{K}x{N}-{seed_tag}", "all")
    outl = synth.outlier_channels(K, rng) if outliers else None
    w = synth.weights(N, K, rng)
    x = synth.activations(M, K, rng, outl)
    b = synth.bias(N, rng) if with_bias else None
    q, s = oracle.quantize_weight(QT[qt], w)
    y = run_w8a16(capi, qt, x, q, s, b)
    if rows is None:
        ref = oracle.w8a16(QT[qt], x, q, s, b)
        return check_tol(y, ref, f"w8a16 {qt} {M}x{K}x{N}")
    ref = oracle.w8a16(QT[qt], x, q, s, b, rows=rows)
    return check_tol(y[rows], ref, f"w8a16 {qt} {M}x{K}x{N} rows")


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M", [1, 2, 3, 8, 16, 17, 31, 64, 127, 129, 255, 256, 257])
def test_w8a16_ragged_m(capi, qt, M):
    w8a16_case(capi, qt, M, 384, 272, True, "ragged-m")


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M,K,N", [(1, 16, 16), (5, 48, 16), (33, 80, 144), (300, 1040, 400), (1024, 512, 384)])
def test_w8a16_ragged_kn(capi, qt, M, K, N):
    w8a16_case(capi, qt, M, K, N, M % 2 == 1, "ragged-kn", outliers=True)


@pytest.mark.parametrize("M,K,N", [(1, 16, 16), (2, 1040, 1040), (3, 18944, 64), (4, 2064, 400), (5, 18944, 64),
                                   (8, 2064, 400), (7, 128, 3584), (13, 528, 2064), (16, 18944, 64),
                                   (17, 3584, 4096), (25, 2064, 400), (32, 3600, 4112), (31, 128, 3584)])
def test_w8a16_e4m3_fp8_path_edges(capi, M, K, N):
    """Up to 32 tokens E4M3 W8A16 runs as FP8 MMAs on the weight codes against
    the activations split into E4M3 terms: every token-tile width (4, 8, 16,
    32) full and with ragged tails, K not a multiple of 128 (and K = 16), N not
    a multiple of the 128-row weight tile, and 1- to 8-way K splits whose
    partial tiles are summed through the cluster's shared memory."""
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A16_LINEAR, "e4m3", M, K, N).startswith("k_w8a16_split+k_w8a16_f8<")
    w8a16_case(capi, "e4m3", M, K, N, M % 2 == 1, "f8", outliers=True)


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M", [1, 32, 128])
def test_w8a16_reads_weights_quantized_just_before(capi, qt, M):
    """Stream order: the weight codes that the kernel right before the linear
    writes on the device (same buffers, no synchronisation in between) are the
    codes the linear reads.  The linears let their weight traffic start during
    the previous kernel's tail; only L2 prefetches run before their wait, so no
    stale code reaches the tensor cores."""
    K, N = 3584, 4096
    rng = synth.rng_for("test-w8a16", 0, f"stream-order-{qt}-{M}", "all")
    w_old, w_new = synth.weights(N, K, rng), synth.weights(N, K, rng)
    x = synth.activations(M, K, rng)
    wd_old, wd_new, xd = to_dev(w_old), to_dev(w_new), to_dev_bf16(x)
    qw = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((N,), dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = capi.workspace(capi.QLIN_OP_W8A16_LINEAR, qt, M, K, N)
    for _ in range(4):
        capi.qlin_quantize_weight(qt, wd_old, qw, s)
        capi.qlin_w8a16_linear(qt, xd, qw, s, None, y, ws)
        capi.qlin_quantize_weight(qt, wd_new, qw, s)
        capi.qlin_w8a16_linear(qt, xd, qw, s, None, y, ws)
    torch.cuda.synchronize()
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    q, sc = oracle.quantize_weight(QT[qt], w_new)
    check_tol(from_dev_bf16(y), oracle.w8a16(QT[qt], x, q, sc, None), f"w8a16 {qt} stream order M={M}")


def test_w8a16_e4m3_fp8_path_wide_dynamic_range(capi):
    """Activations spanning 2^16 within a row: the two-band split keeps every
    element within 2^-28.8 of the row's maximum exactly."""
    M, K, N = 8, 2048, 1024
    rng = synth.rng_for("test-w8a16", 0, "f8-range", "all")
    w = synth.weights(N, K, rng)
    xf = synth.bf16_bits_to_f32(synth.activations(M, K, rng))
    xf = xf * np.exp2(rng.integers(-16, 1, size=xf.shape)).astype(np.float32)
    x = synth.f32_to_bf16_bits(xf)
    q, s = oracle.quantize_weight(oracle.E4M3, w)
    y = run_w8a16(capi, "e4m3", x, q, s, None)
    check_tol(y, oracle.w8a16(oracle.E4M3, x, q, s, None), "w8a16 e4m3 wide range")


def _massive_case(capi, name, M, magnitude, zero_weights, tag):
    lin = [l for l in synth.workload(synth.DECODE7B).linears if l.name == name and l.M == 1][0]
    K, N = lin.K, lin.N
    rng = synth.rng_for("test-w8a16", 0, f"massive-{name}-{M}-{magnitude}-{zero_weights}-{tag}", "all")
    w = synth.weights(N, K, rng)
    xf = synth.bf16_bits_to_f32(synth.activations(M, K, rng, synth.outlier_channels(K, rng)))
    massive = rng.choice(K, size=4, replace=False)
    sign = np.where(rng.random((M, 4)) < 0.5, -1.0, 1.0).astype(np.float32)
    xf[:, massive] = sign * np.float32(magnitude) * (1.0 + rng.random((M, 4))).astype(np.float32)
    if zero_weights:
        w[:, massive] = 0.0
    x = synth.f32_to_bf16_bits(xf)
    q, s = oracle.quantize_weight(oracle.E4M3, w)
    assert "k_w8a16_f8<" in capi.qlin_kernel_name(capi.QLIN_OP_W8A16_LINEAR, "e4m3", M, K, N)
    y = run_w8a16(capi, "e4m3", x, q, s, None)
    return check_tol(y, oracle.w8a16(oracle.E4M3, x, q, s, None), f"massive {name} M={M} 2^{np.log2(magnitude):.0f}")


@pytest.mark.parametrize("M", [1, 8, 32])
@pytest.mark.parametrize("name", ["q_proj", "gate_up_proj", "down_proj"])
def test_w8a16_e4m3_massive_activations_zero_weights(capi, name, M):
    """Rows with "massive activations": four channels 2^20 above the rest (N(0,1)
    plus 1 % outlier channels x20) whose weight codes are all zero, so the
    ordinary elements alone decide y.  The split's band B holds every ordinary
    element exactly; with band A alone they would keep only about two bits."""
    _massive_case(capi, name, M, 2.0 ** 20, True, "z20")


@pytest.mark.parametrize("M", [1, 32])
@pytest.mark.parametrize("magnitude", [2.0 ** 10, 2.0 ** 14, 2.0 ** 18])
def test_w8a16_e4m3_massive_activations_span(capi, M, magnitude):
    """Massive channels from 2^10 to 2^18 above the rest, zero weights on them."""
    _massive_case(capi, "q_proj", M, magnitude, True, "span")


@pytest.mark.parametrize("M", [1, 32])
def test_w8a16_e4m3_massive_activations_live_weights(capi, M):
    """Massive channels 2^18 above the rest with ordinary weights: y is dominated
    by them and still within tolerance."""
    _massive_case(capi, "q_proj", M, 2.0 ** 18, False, "live")


def test_w8a16_e4m3_split_exact_window(capi):
    """Ordinary elements spread over 28 binades (N(0,1) times 2^U(-28, 0)), and
    channel 0 at 448 * 2^-r in row r, so the rows' scales and the place of
    their elements in the two bands vary row by row; every element within
    2^-28.8 of its row's maximum is represented exactly."""
    M, K, N = 24, 2048, 512
    rng = synth.rng_for("test-w8a16", 0, "f8-window", "all")
    w = synth.weights(N, K, rng)
    xf = synth.bf16_bits_to_f32(synth.activations(M, K, rng))
    xf = xf * np.exp2(rng.uniform(-28.0, 0.0, size=xf.shape)).astype(np.float32)
    xf[:, 0] = np.float32(448.0) * np.exp2(-np.arange(M, dtype=np.float32))
    x = synth.f32_to_bf16_bits(xf)
    q, s = oracle.quantize_weight(oracle.E4M3, w)
    y = run_w8a16(capi, "e4m3", x, q, s, None)
    check_tol(y, oracle.w8a16(oracle.E4M3, x, q, s, None), "w8a16 e4m3 exact window")


@pytest.mark.parametrize("M", [1, 16])
def test_w8a16_int8_small_workload(capi, M):
    """INT8 W8A16 single linear K=N=1024, M in {1,16}, full output checked."""
    lin = [l for l in synth.workload(synth.SMALL).linears if l.M == M][0]
    t, q, s = _operands(lin)
    y = run_w8a16(capi, "int8", t["x"], q, s, None)
    check_tol(y, oracle.w8a16(oracle.INT8, t["x"], q, s), f"small M={M}")


@pytest.mark.parametrize("M", [1, 8, 32, 128, 256])
@pytest.mark.parametrize("name", ["q_proj", "gate_up_proj", "down_proj"])
def test_w8a16_decode7b_full_size(capi, name, M):
    """FP8-E4M3 W8A16 decode sweep at full size, sampled output rows."""
    lin = [l for l in synth.workload(synth.DECODE7B).linears if l.name == name and l.M == M][0]
    t, q, s = _operands(lin)
    y = run_w8a16(capi, "e4m3", t["x"], q, s, None)
    rows = sample_rows(M, 8)
    check_tol(y[rows], oracle.w8a16(oracle.E4M3, t["x"], q, s, rows=rows), f"{name} M={M}")


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_w8a16_zero_weight_gives_bias(capi, qt):
    M, K, N = 5, 64, 48
    rng = np.random.default_rng(0)
    b = synth.bias(N, rng)
    x = synth.activations(M, K, rng)
    q, s = oracle.quantize_weight(QT[qt], np.zeros((N, K), np.float32))
    y = run_w8a16(capi, qt, x, q, s, b)
    assert np.array_equal(y, np.broadcast_to(b, (M, N)))


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_w8a16_power_of_two_scaling_bitexact(capi, qt):
    """W * 2^j: same codes, scales * 2^j, so the BF16 output scales bit-exactly."""
    M, K, N = 9, 256, 128
    rng = np.random.default_rng(3)
    w = synth.weights(N, K, rng)
    x = synth.activations(M, K, rng)
    q1, s1 = oracle.quantize_weight(QT[qt], w)
    q2, s2 = oracle.quantize_weight(QT[qt], w * np.float32(16))
    assert np.array_equal(q1, q2)
    y1 = synth.bf16_bits_to_f32(run_w8a16(capi, qt, x, q1, s1, None))
    y2 = synth.bf16_bits_to_f32(run_w8a16(capi, qt, x, q2, s2, None))
    assert np.array_equal(y2, y1 * np.float32(16))


def test_w8a16_m0_is_noop(capi):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    qw = torch.zeros((32, 64), dtype=torch.uint8, device="cuda")
    s = torch.ones(32, device="cuda")
    y = capi.w8a16_linear("int8", x, qw, s)
    assert y.shape == (0, 32)


# ------------------------------------------------------------------ W8A8
def w8a8_case(capi, qt, M, K, N, with_bias, tag, rows=None, outliers=False):
    rng = synth.rng_for("test-w8a8", 0, f"{qt}-{M}x{K}x{N}-{tag}", "all")
    outl = synth.outlier_channels(K, rng) if outliers else None
    w = synth.weights(N, K, rng)
    cal = synth.activations(1024, K, rng, outl)
    x = synth.activations(M, K, rng, outl)
    b = synth.bias(N, rng) if with_bias else None
    q, s = oracle.quantize_weight(QT[qt], w)
    sx = oracle.act_scale(QT[qt], cal)
    y = run_w8a8(capi, qt, x, sx, q, s, b)
    qx = oracle.quantize_act(QT[qt], x, sx)
    ref = oracle.w8a8(QT[qt], qx, sx, q, s, b, rows=rows)
    return check_tol(y if rows is None else y[rows], ref, f"w8a8 {qt} {M}x{K}x{N}")


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M", [1, 3, 16, 127, 129, 256, 257, 1024])
def test_w8a8_ragged_m(capi, qt, M):
    w8a8_case(capi, qt, M, 512, 272, True, "ragged-m", outliers=True)


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M,K,N", [(1, 16, 16), (7, 48, 32), (130, 1040, 400), (2048, 2048, 512)])
def test_w8a8_ragged_kn(capi, qt, M, K, N):
    w8a8_case(capi, qt, M, K, N, M % 2 == 0, "ragged-kn")


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_w8a8_int8_3b_workload(capi, idx):
    """INT8 W8A8 static on the 3B microbench shapes with bias, full size, full output."""
    lin = synth.workload(synth.W8A8_3B).linears[idx]
    t, q, s = _operands(lin)
    sx = oracle.act_scale(oracle.INT8, t["cal"])
    y = run_w8a8(capi, "int8", t["x"], sx, q, s, t["bias"])
    rows = None if lin.M <= 256 else sample_rows(lin.M, 32)
    qx = oracle.quantize_act(oracle.INT8, t["x"], sx)
    ref = oracle.w8a8(oracle.INT8, qx, sx, q, s, t["bias"], rows=rows)
    check_tol(y if rows is None else y[rows], ref, f"3b {lin.name} M={lin.M}")


@pytest.mark.parametrize("M", [1024, 4096, 16384, 32640])
@pytest.mark.parametrize("K,N", [(2048, 11008), (11008, 2048), (2048, 2048)])
def test_w8a8_e4m3_prefill(capi, M, K, N):
    """FP8-E4M3 W8A8 static prefill workload, every shape at full size, sampled
    output rows.  K = 11008 -> 2048 from 16384 tokens on takes the GEMM that
    quantizes its activations itself; the other shapes quantize in a separate
    pass."""
    lin = [l for l in synth.workload(synth.PREFILL).linears if l.M == M and l.K == K and l.N == N][0]
    fused = M >= 16384 and K == 11008
    assert capi.qlin_kernel_name(capi.QLIN_OP_W8A8_LINEAR, "e4m3", M, K, N) == \
        ("k_fp8_gemm<xq>" if fused else "k_quantize_act+k_fp8_gemm")
    t, q, s = _operands(lin)
    sx = oracle.act_scale(oracle.E4M3, t["cal"])
    y = run_w8a8(capi, "e4m3", t["x"], sx, q, s, None)
    rows = sample_rows(M, 24)
    qx = oracle.quantize_act(oracle.E4M3, t["x"][rows], sx)
    ref = oracle.w8a8(oracle.E4M3, qx, sx, q, s)
    check_tol(y[rows], ref, f"prefill {M}x{K}x{N}")


# ------------------------------------------- 36-layer 3B stack, unmerged
STACK_SHAPES = [("q_proj", 2048, 2048), ("k_proj", 2048, 256), ("gate_up_proj", 2048, 22016),
                ("down_proj", 11008, 2048)]  # o_proj is q_proj's shape, v_proj k_proj's


@pytest.mark.parametrize("name,K,N", STACK_SHAPES)
def test_stack_decode_int8_w8a16(capi, name, K, N):
    """The 3B stack's decode linears (INT8 W8A16, 256 tokens), layer 0's
    tensors, sampled output rows."""
    lin = [l for l in synth.stack_linears("decode") if l.layer == 0 and l.name == name][0]
    assert (lin.K, lin.N, lin.M) == (K, N, 256)
    t, q, s = _operands(lin)
    y = run_w8a16(capi, "int8", t["x"], q, s, None)
    rows = sample_rows(lin.M, 32)
    check_tol(y[rows], oracle.w8a16(oracle.INT8, t["x"], q, s, rows=rows), f"stack decode {name}")


@pytest.mark.parametrize("name,K,N", STACK_SHAPES)
def test_stack_prefill_e4m3_w8a8(capi, name, K, N):
    """The 3B stack's prefill linears (E4M3 W8A8 static, 8192 tokens), layer
    0's tensors, sampled output rows."""
    lin = [l for l in synth.stack_linears("prefill") if l.layer == 0 and l.name == name][0]
    assert (lin.K, lin.N, lin.M) == (K, N, 8192)
    t, q, s = _operands(lin)
    sx = oracle.act_scale(oracle.E4M3, t["cal"])
    y = run_w8a8(capi, "e4m3", t["x"], sx, q, s, None)
    rows = sample_rows(lin.M, 24)
    ref = oracle.w8a8(oracle.E4M3, oracle.quantize_act(oracle.E4M3, t["x"][rows], sx), sx, q, s)
    check_tol(y[rows], ref, f"stack prefill {name}")


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_w8a8_zero_weight_gives_bias(capi, qt):
    M, K, N = 6, 64, 32
    rng = np.random.default_rng(4)
    b = synth.bias(N, rng)
    x = synth.activations(M, K, rng)
    q, s = oracle.quantize_weight(QT[qt], np.zeros((N, K), np.float32))
    y = run_w8a8(capi, qt, x, np.float32(0.05), q, s, b)
    assert np.array_equal(y, np.broadcast_to(b, (M, N)))


# ----------------------------------------------------- INT8 accumulator
@pytest.mark.parametrize("M,K,N", [(1, 16, 16), (3, 48, 32), (127, 1040, 144), (256, 11008, 2048),
                                   (1024, 2048, 1024)])
def test_i8_gemm_bitexact(capi, M, K, N):
    rng = np.random.default_rng(M * 7 + K)
    qx = rng.integers(-127, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    acc = capi.i8_gemm_s32(to_dev(qx.view(np.uint8)), to_dev(qw.view(np.uint8))).cpu().numpy()
    assert np.array_equal(acc, oracle.i8_gemm(qx, qw))


def test_i8_gemm_worst_case_magnitude(capi):
    """All +-127 at K=18944: |acc| = 127*127*18944, the largest the layer meets."""
    K = 18944
    qx = np.full((130, K), 127, np.int8)
    qx[1::2] = -127
    qw = np.full((144, K), 127, np.int8)
    qw[::3] = -127
    acc = capi.i8_gemm_s32(to_dev(qx.view(np.uint8)), to_dev(qw.view(np.uint8))).cpu().numpy()
    ref = oracle.i8_gemm(qx, qw)
    assert np.abs(ref).max() == 127 * 127 * K
    assert np.array_equal(acc, ref)


def test_i8_gemm_one_hot(capi):
    rng = np.random.default_rng(12)
    M, K, N = 40, 256, 64
    qx = rng.integers(-127, 128, (M, K), dtype=np.int8)
    perm = rng.permutation(K)[:N]
    qw = np.zeros((N, K), np.int8)
    qw[np.arange(N), perm] = 127
    acc = capi.i8_gemm_s32(to_dev(qx.view(np.uint8)), to_dev(qw.view(np.uint8))).cpu().numpy()
    assert np.array_equal(acc, 127 * qx[:, perm].astype(np.int32))


# ------------------------------------------------------ failure detection
def test_bounded_wait_reports_timeout(capi):
    flag = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    capi.qlin_debug_wait_flag(flag, 2_000_000)  # nothing sets the flag: gives up after 2 ms
    assert capi.qlin_get_device_status() == capi.QLIN_ERR_TIMEOUT
    assert capi.qlin_get_device_status() == capi.QLIN_OK  # cleared by the read
    flag.fill_(1)
    capi.qlin_debug_wait_flag(flag, 2_000_000)
    assert capi.qlin_get_device_status() == capi.QLIN_OK
    y = capi.w8a16_linear("int8", torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda"),
                          torch.zeros((16, 64), dtype=torch.uint8, device="cuda"), torch.ones(16, device="cuda"))
    torch.cuda.synchronize()  # the context is still usable
    assert y.float().abs().sum().item() == 0.0


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M,K,N", [(64, 1040, 1024), (100, 2048, 1024), (200, 1040, 2048), (256, 3584, 4096),
                                   (700, 2048, 2048), (1024, 1024, 4096)])
def test_w8a16_split_k_cluster_shapes(capi, qt, M, K, N):
    """Shapes with few output tiles, whose K range is split over the CTAs of a
    cluster (the partial tiles are summed through distributed shared memory),
    and shapes past the 128-token tile; ragged M and K included."""
    rows = None if M <= 256 else sample_rows(M, 24)
    w8a16_case(capi, qt, M, K, N, True, "splitk", rows=rows, outliers=True)


@pytest.mark.parametrize("M,K,N", [(64, 1040, 1024), (200, 2048, 2048)])
def test_i8_gemm_split_k_bitexact(capi, M, K, N):
    rng = np.random.default_rng(M + K + N)
    qx = rng.integers(-127, 128, (M, K), dtype=np.int8)
    qw = rng.integers(-127, 128, (N, K), dtype=np.int8)
    acc = capi.i8_gemm_s32(to_dev(qx.view(np.uint8)), to_dev(qw.view(np.uint8))).cpu().numpy()
    assert np.array_equal(acc, oracle.i8_gemm(qx, qw))


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
def test_w8a16_reads_every_weight_code_exactly(capi, qt):
    """Every 8-bit weight code, including the E4M3 subnormals, negative zero and the
    saturation codes, through the W8A16 linear: with one-hot activations and unit
    scales, y[m, n] is the exact value of code q[n, m] (each is a BF16 number)."""
    codes = np.array([c for c in range(256) if qt == "int8" or (c & 0x7F) != 0x7F], np.uint8)
    if qt == "int8":
        codes = codes[codes != 0x80]  # -128 is never produced
    N = 256
    K = int(np.ceil(len(codes) / 16.0) * 16)
    q = np.zeros((N, K), np.uint8)
    rng = np.random.default_rng(9)
    for n in range(N):
        q[n, :len(codes)] = rng.permutation(codes)
    M = K
    x = synth.f32_to_bf16_bits(np.eye(M, K, dtype=np.float32))  # token m selects column m
    s = np.ones(N, np.float32)
    y = synth.bf16_bits_to_f32(run_w8a16(capi, qt, x, q, s, None)).astype(np.float64)
    if qt == "int8":
        want = q.view(np.int8).astype(np.float64).T
    else:
        table = np.array([oracle.e4m3_decode(c) for c in range(256)])
        want = table[q].T
    assert np.array_equal(y, want[:M]), int((y != want[:M]).sum())


@pytest.mark.parametrize("qt", ["int8", "e4m3"])
@pytest.mark.parametrize("M,K,N", [(256, 1024, 22016), (200, 2048, 19712)])
def test_w8a16_partial_last_wave(capi, qt, M, K, N):
    """More weight-tile units than SMs with a mostly empty last wave (344 units
    of 128 x 128 at 256 tokens; 308 at 200 tokens, a ragged token tile): the
    persistent CTAs take three units or two.  Full output against the oracle."""
    w8a16_case(capi, qt, M, K, N, M % 2 == 0, "last-wave")
