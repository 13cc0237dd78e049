/*
 * qlin.h -- C ABI of libqlin, an 8-bit quantized linear layer for GB300 (sm_103a).
 *
 * Two forms of the layer, as the serving pages describe them:
 *   W8A16 weight-only: 8-bit weights (INT8 or OCP FP8-E4M3) with one scale per
 *     output channel, BF16 activations; the weights are dequantized to BF16 and
 *     a standard matmul with fp32 accumulation follows ("Nano-vLLM-MoE" README,
 *     "FP8 W8A16 weight-only quantization", Setup; "Nano-vLLM-MOE" README,
 *     "INT8 量化支持", list "关键设计", W8A16 item).
 *   W8A8 static: activations are quantized with one offline-calibrated
 *     per-tensor input_scale, then an 8-bit GEMM runs with a scale epilogue
 *     ("Nano-vLLM-MOE" README, "INT8 量化支持", "关键设计", W8A8 static item;
 *     "Nano-vLLM-MoE" README, "FP8 W8A8 static quantization", Setup:
 *     offline-calibrated activation scales, linear backends with a custom
 *     epilogue).
 * The per-output-channel granularity, scale = max|row|/127 (INT8) or /448
 * (E4M3), the symmetric clamp to [-127,127] and the saturating E4M3 cast are
 * this layer's stated definition; the pages only name the schemes.
 *
 * Conventions for every entry point:
 *   - Layouts are row-major and dense: x [M,K] BF16, W / qw [N,K] (nn.Linear,
 *     K contiguous), y [M,N] BF16, w_scale [N] fp32, bias [N] BF16.
 *     BF16 data is passed as raw 16-bit patterns (uint16_t storage).
 *   - All data pointers are DEVICE pointers into memory the caller owns.  The
 *     library allocates no device memory on these paths; where an operation
 *     needs scratch it takes a caller-owned workspace (`ws`, `ws_bytes`) whose
 *     size qlin_workspace_bytes() reports.  Nothing is retained between calls.
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream) and
 *     returns once the work is enqueued.  Only qlin_get_device_status()
 *     synchronizes.
 *   - Calls on one stream are ordered like any work on it.  A call sees
 *     everything earlier work on the stream wrote, weights included, and
 *     later work sees its outputs.  Consecutive kernels of the library start
 *     early (programmatic dependent launch): a kernel's CTAs take SMs while its
 *     predecessor finishes, and wait for it before they read its outputs.  The
 *     inputs read before that wait are a linear's weights: its codes (`qw`),
 *     their scales (`w_scale`) and its bias.  So none of these may be the
 *     output of the library call right before the linear on its stream, other
 *     than qlin_quantize_weight (which lets no later kernel start before it
 *     completes).  Weights written by any other kernel or copy, or by any
 *     earlier call, are read as written.
 *   - Argument errors are detected on the host before anything is launched and
 *     returned as a status: NULL required pointer, negative sizes, K or N not a
 *     multiple of 16, pointers not 16-byte aligned, unknown qtype, workspace
 *     too small.  A CUDA launch error is returned as QLIN_ERR_CUDA.  No entry
 *     point aborts, traps or throws across the ABI.
 *   - M == 0 is valid and enqueues nothing.
 *   - Device-side waits in the kernels are bounded; a wait that runs out sets
 *     a device status word instead of hanging, which qlin_get_device_status()
 *     reports as QLIN_ERR_TIMEOUT.  A kernel whose cluster shape is not the
 *     one it was launched for (a tool that re-issues the launch without it)
 *     does no work and sets QLIN_ERR_UNSUPPORTED there.
 */
#ifndef QLIN_H_
#define QLIN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle; identical to cudaStream_t / CUstream. */
typedef struct CUstream_st *qlin_stream_t;

typedef enum {
  QLIN_OK = 0,
  QLIN_ERR_INVALID_ARG = 1, /* NULL pointer, bad size, misalignment, K/N % 16 != 0 */
  QLIN_ERR_UNSUPPORTED = 2, /* no device, not sm_103, qtype not valid here, or
                               (device status) a kernel launched without its
                               cluster shape */
  QLIN_ERR_WORKSPACE = 3,   /* ws NULL or ws_bytes < qlin_workspace_bytes() */
  QLIN_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  QLIN_ERR_TIMEOUT = 5      /* a bounded device-side wait ran out (device status) */
} qlin_status;

typedef enum {
  QLIN_INT8 = 0, /* signed 8-bit integer codes in [-127, 127] */
  QLIN_E4M3 = 1  /* OCP FP8 E4M3 ("e4m3fn"): bias 7, no inf, max finite 448 */
} qlin_qtype;

typedef enum {
  QLIN_OP_QUANTIZE_WEIGHT = 0,
  QLIN_OP_ACT_SCALE = 1,
  QLIN_OP_QUANTIZE_ACT = 2,
  QLIN_OP_W8A16_LINEAR = 3,
  QLIN_OP_W8A8_LINEAR = 4,
  QLIN_OP_I8_GEMM_S32 = 5,
  QLIN_OP_W8A8_DYNAMIC_LINEAR = 6,
  QLIN_OP_KV_STORE_MIXED = 7, /* for qlin_kernel_name: M = tokens, K = head_dim, N = kv heads */
  QLIN_OP_KV_LOAD_MIXED = 8,
  QLIN_OP_W8A16_GATE_UP_SILU = 9, /* N = the intermediate size I (output channels) */
  QLIN_OP_W8A8_GATE_UP_SILU = 10
} qlin_op;

/*
 * Per-output-channel symmetric weight quantization (offline export step;
 * "Nano-vLLM-MOE" README, "INT8 量化支持", 快速使用 step 1 `--scheme int8_w8a16`;
 * "Nano-vLLM-MoE" README, FP8 W8A16 Setup, `--scheme fp8_w8a16` export).
 *   w        [N,K] fp32 input weights (device, read only).
 *   qw       [N,K] 1-byte output codes (device): int8 two's complement for
 *            QLIN_INT8, E4M3 bit patterns for QLIN_E4M3.
 *   w_scale  [N] fp32 output scales (device).
 * Computes, per row n:  s = max_k |w[n,k]| / QMAX  (QMAX = 127 or 448, one IEEE
 * binary32 division; s = 1 for an all-zero row), then for every k
 *   v = w[n,k] / s (IEEE binary32 division) and
 *   INT8: q = clamp(round_half_even(v), -127, 127);
 *   E4M3: q = nearest E4M3 value (ties to even), |v| > 448 saturates to +-448.
 * Requirements: N >= 0, K >= 16, K % 16 == 0, all pointers 16-byte aligned.
 */
qlin_status qlin_quantize_weight(qlin_qtype qtype, int64_t N, int64_t K, const float *w,
                                 void *qw, float *w_scale, qlin_stream_t stream);

/*
 * Static per-tensor activation scale from a calibration batch (offline
 * calibration; "Nano-vLLM-MOE" README, "INT8 量化支持", 关键设计 W8A8 static
 * item: offline per-layer input_scale; 快速使用 step 2:
 * `--calib-samples 64 --calib-seqlen 512`).
 *   x_cal        [rows,K] BF16 calibration activations (device).
 *   input_scale  one fp32 output on the device: max|x_cal| / QMAX, or 1 when the
 *                batch is all zero.
 *   ws           device workspace of qlin_workspace_bytes(QLIN_OP_ACT_SCALE, ...)
 *                bytes (4 bytes today, 256-byte aligned); overwritten.
 * Requirements: rows >= 1, K >= 16, K % 16 == 0, pointers 16-byte aligned.
 */
qlin_status qlin_act_scale_from_calib(qlin_qtype qtype, int64_t rows, int64_t K,
                                      const void *x_cal, float *input_scale, void *ws,
                                      size_t ws_bytes, qlin_stream_t stream);

/*
 * Static activation quantization with the fixed calibrated scalar
 * ("Nano-vLLM-MOE" README, "INT8 量化支持", 关键设计 W8A8 static item:
 * quantize activations at run time with the fixed scalar).
 *   x            [M,K] BF16 (device).
 *   input_scale  one fp32 on the device (so the call can sit in a CUDA graph).
 *   qx           [M,K] 1-byte output codes (device):
 *                INT8: clamp(round_half_even(x / s), -127, 127)
 *                E4M3: saturating round-half-even E4M3 cast of x / s.
 * Requirements: M >= 0, K >= 16, K % 16 == 0, pointers 16-byte aligned.
 */
qlin_status qlin_quantize_act_static(qlin_qtype qtype, int64_t M, int64_t K, const void *x,
                                     const float *input_scale, void *qx, qlin_stream_t stream);

/*
 * W8A16 weight-only linear ("Nano-vLLM-MoE" README, FP8 W8A16 Setup: FP8->BF16
 * dequant GEMM, bf16 x bf16 with fp32 accumulation; "Nano-vLLM-MOE" README,
 * 关键设计 W8A16 item: INT8 weights dequantized to BF16 for a standard matmul):
 *   y[m,n] = bf16( w_scale[n] * sum_k x[m,k] * deq(qw[n,k]) + bias[n] )
 * deq() is exact (every INT8 and E4M3 value is a BF16 value); the per-channel
 * scale factors out of the k-sum and is applied in fp32 in the epilogue;
 * accumulation is fp32; the output is rounded to BF16 (nearest even).
 *   x [M,K] BF16, qw [N,K] codes, w_scale [N] fp32, bias [N] BF16 or NULL,
 *   y [M,N] BF16 output.  ws/ws_bytes: workspace of
 *   qlin_workspace_bytes(QLIN_OP_W8A16_LINEAR, ...) bytes (may be NULL when that is 0).
 * Requirements: M >= 0, K >= 16, N >= 16, K % 16 == 0, N % 16 == 0, pointers
 * 16-byte aligned, y must not overlap any input.
 */
qlin_status qlin_w8a16_linear(qlin_qtype qtype, int64_t M, int64_t K, int64_t N, const void *x,
                              const void *qw, const float *w_scale, const void *bias, void *y,
                              void *ws, size_t ws_bytes, qlin_stream_t stream);

/*
 * W8A8 static linear ("Nano-vLLM-MOE" README, 关键设计 W8A8 static item;
 * "Nano-vLLM-MoE" README, FP8 W8A8 static Setup: 8-bit GEMM + custom epilogue):
 *   qx = quantize_act_static(x, input_scale)           (into the workspace)
 *   acc[m,n] = sum_k deq(qx[m,k]) * deq(qw[n,k])       (INT8: exact int32;
 *                                                        E4M3: fp32 accumulate)
 *   y[m,n] = bf16( acc * (input_scale * w_scale[n]) + bias[n] )
 * The INT8 accumulator is exact for every input (|acc| <= 127*127*K < 2^31).
 *   x [M,K] BF16, input_scale fp32 scalar (device), qw [N,K] codes of the same
 *   qtype, w_scale [N], bias [N] BF16 or NULL, y [M,N] BF16.
 *   ws: qlin_workspace_bytes(QLIN_OP_W8A8_LINEAR, qtype, M, K, N) bytes.
 * Requirements as for qlin_w8a16_linear.
 * Execution: for E4M3 with at least 16 token tiles of 128 and N <= 4096 the
 * quantization runs inside the GEMM kernel (a cooperative launch of 2-CTA
 * clusters); the codes still land in the workspace.  QLIN_FP8_FUSED_QUANT=0 in
 * the environment (read once per process) selects the separate quantization
 * pass instead, e.g. under a profiler that re-issues cooperative launches
 * without their cluster shape (the fused kernel would report
 * QLIN_ERR_UNSUPPORTED there).  Same results either way.
 */
qlin_status qlin_w8a8_linear(qlin_qtype qtype, int64_t M, int64_t K, int64_t N, const void *x,
                             const float *input_scale, const void *qw, const float *w_scale,
                             const void *bias, void *y, void *ws, size_t ws_bytes,
                             qlin_stream_t stream);

/*
 * Dynamic per-token activation quantization: the per-token abs-max scheme that
 * "Nano-vLLM-MOE" README ("INT8 量化支持", 关键设计, W8A8 static item) contrasts
 * with the static scalar (it costs one more reduction per token).  Per row m:
 *   x_scale[m] = max_k |x[m,k]| / QMAX  (IEEE binary32 division; 1 for a zero row)
 *   qx[m,k]    = INT8: clamp(round_half_even(x[m,k] / x_scale[m]), -127, 127)
 *                E4M3: saturating round-half-even E4M3 cast of x[m,k] / x_scale[m]
 *   x [M,K] BF16, qx [M,K] 1-byte codes, x_scale [M] fp32 (all device).
 * Requirements: M >= 0, K >= 16, K % 16 == 0, pointers 16-byte aligned.
 */
qlin_status qlin_quantize_act_dynamic(qlin_qtype qtype, int64_t M, int64_t K, const void *x, void *qx,
                                      float *x_scale, qlin_stream_t stream);

/*
 * W8A8 linear with dynamic per-token activation scales (same reading as above):
 *   qx, s_x = quantize_act_dynamic(x)                    (into the workspace)
 *   y[m,n]  = bf16( acc[m,n] * (s_x[m] * w_scale[n]) + bias[n] )
 * with acc as in qlin_w8a8_linear (exact int32 for INT8, fp32 for E4M3).
 *   ws: qlin_workspace_bytes(QLIN_OP_W8A8_DYNAMIC_LINEAR, qtype, M, K, N) bytes.
 * Requirements as for qlin_w8a16_linear.
 */
qlin_status qlin_w8a8_dynamic_linear(qlin_qtype qtype, int64_t M, int64_t K, int64_t N, const void *x,
                                     const void *qw, const float *w_scale, const void *bias, void *y, void *ws,
                                     size_t ws_bytes, qlin_stream_t stream);

/*
 * Raw INT8 GEMM accumulator, the integer core of the INT8 W8A8 linear, exposed
 * so it can be checked bit for bit: acc[m,n] = sum_k qx[m,k] * qw[n,k] (int32).
 *   qx [M,K] int8, qw [N,K] int8, acc [M,N] int32 (device).
 *   ws: qlin_workspace_bytes(QLIN_OP_I8_GEMM_S32, QLIN_INT8, M, K, N) bytes.
 * Requirements as for qlin_w8a16_linear.
 */
qlin_status qlin_i8_gemm_s32(int64_t M, int64_t K, int64_t N, const void *qx, const void *qw,
                             int32_t *acc, void *ws, size_t ws_bytes, qlin_stream_t stream);

/*
 * W8A8 static linear for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for callers
 * that run where cudaMalloc (and any allocating library, torch included) is not
 * available or not allowed: inference plugins handed a fixed memory budget,
 * code enqueued while a stream is being captured into a CUDA graph, or
 * runtimes that must not grow device memory after start-up.  It computes
 * exactly what qlin_w8a8_linear computes (the same kernels on the same
 * inputs, so the same bits), with the same arguments minus the workspace: the
 * quantized activations (and, for large E4M3 calls, the task flags of the
 * fused-quantization GEMM) go to a scratch array that the library holds in
 * device memory of its own (a file-scope __device__ array of
 * QLIN_W8A8_NOALLOC_SCRATCH_BYTES bytes, 64 MiB, which every GPU that loads
 * the library keeps until the process exits).
 *   - Argument errors are reported exactly as qlin_w8a8_linear reports them,
 *     from the same checks in the same order: arguments, then size, then the
 *     device (QLIN_ERR_UNSUPPORTED on a GPU other than sm_103a).
 *   - Sizes whose workspace (qlin_workspace_bytes(QLIN_OP_W8A8_LINEAR, qtype,
 *     M, K, N)) exceeds QLIN_W8A8_NOALLOC_SCRATCH_BYTES are rejected with
 *     QLIN_ERR_WORKSPACE before anything is launched.
 *   - The first call with M > 0 on a device looks up the scratch array's
 *     device address (once per device, with that device current); make that
 *     first call before any stream capture begins.
 *   - Every call on a device shares the one scratch array, which keeps what the
 *     last call left there.  A call reads only what it has written itself; the
 *     task flags that must start at zero are cleared by the call, on its
 *     stream, before its GEMM runs.  Calls that can overlap on the GPU
 *     (different streams without ordering) race on the array; order them.
 * It calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define QLIN_W8A8_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
qlin_status qlin_w8a8_linear_noalloc(qlin_qtype qtype, int64_t M, int64_t K, int64_t N, const void *x,
                                     const float *input_scale, const void *qw, const float *w_scale,
                                     const void *bias, void *y, qlin_stream_t stream);

/*
 * Merged gate_up linear with the SiLU * up epilogue.  The "tiny-vLLM" README's
 * quality check counts four quantized linears per layer of its 28-layer model
 * (112 target layers): merged qkv, o, merged gate_up and down.  The model
 * family's MLP is down(silu(gate(x)) * up(x)); these entry points compute the
 * merged gate_up linear and its activation in one kernel, so the [M, 2I]
 * intermediate never reaches memory:
 *   qw [2I, K] codes with the gate rows [0, I) above the up rows [I, 2I)
 *   (the export layout of a merged gate_up projection), w_scale [2I] fp32,
 *   bias [2I] BF16 or NULL;
 *   g = the linear's fp32 output for row n, u = for row I + n (bias added),
 *   y[m, n] = bf16( silu(g) * u ),  silu(g) = g / (1 + exp(-g)),  y [M, I].
 * g and u are not rounded to BF16 in between.  I must be a multiple of 128.
 * qlin_w8a16_gate_up_silu takes BF16 x like qlin_w8a16_linear (no workspace);
 * qlin_w8a8_gate_up_silu quantizes x with the static input_scale like
 * qlin_w8a8_linear (workspace: qlin_workspace_bytes(QLIN_OP_W8A8_GATE_UP_SILU,
 * qtype, M, K, I) bytes).  Other requirements as for those linears.
 * The merged qkv linear needs no entry point of its own: its per-channel
 * scales make it qlin_w8a16_linear / qlin_w8a8_linear over the concatenated
 * weight [Nq + Nk + Nv, K].
 */
qlin_status qlin_w8a16_gate_up_silu(qlin_qtype qtype, int64_t M, int64_t K, int64_t I, const void *x,
                                    const void *qw, const float *w_scale, const void *bias, void *y, void *ws,
                                    size_t ws_bytes, qlin_stream_t stream);
qlin_status qlin_w8a8_gate_up_silu(qlin_qtype qtype, int64_t M, int64_t K, int64_t I, const void *x,
                                   const float *input_scale, const void *qw, const float *w_scale,
                                   const void *bias, void *y, void *ws, size_t ws_bytes, qlin_stream_t stream);

/*
 * Mixed KV-cache quantization ("Nano-vLLM-MoE" README, section "KV cache
 * compression": mixed K int8 + V FP8, K group 32, float16 scales; Highlights:
 * dynamic per-token quantization; the layout below is the one whose size is
 * the printed 0.5195x BF16 bytes per block).  A cache of num_slots slots (a
 * slot is block * block_size + offset in a paged cache), H kv heads and
 * head_dim D in {32, 64, 128, 256}, four device arrays the caller owns:
 *   k_cache [num_slots, H, D]     int8 codes
 *   k_scale [num_slots, H, D/32]  float16 bits, one per 32 consecutive elements
 *   v_cache [num_slots, H, D]     E4M3 codes
 *   v_scale [num_slots, H]        float16 bits, one per (slot, head)
 *
 * qlin_kv_store_mixed quantizes the T new tokens and writes them to their
 * slots.  For token t with slot = slots[t] >= 0 and each head h:
 *   key group g (elements 32g..32g+31):
 *     s = RN_fp16(fl32(max|k| / 127)), saturating at 65504; 1.0 if that is 0
 *     k_cache = clamp(rint(fl32(k / s)), -127, 127)   (round half to even)
 *   value head:
 *     s = RN_fp16(fl32(max|v| / 448)), same rules
 *     v_cache = saturating RNE E4M3 cast of fl32(v / s)
 *   k, v: BF16 [T, ld] device rows; token t's H*D elements (head-major) start
 *     at k + t*ldk (v + t*ldv); ldk, ldv >= H*D and multiples of 8, so the key
 *     and value columns of a fused QKV output can be passed in place.
 *   slots: int64 [T] device array.  A negative slot skips the token (padding).
 *     A slot >= num_slots breaks the contract: the token is skipped and the
 *     device status word is set to QLIN_ERR_INVALID_ARG (reported by
 *     qlin_get_device_status).  Two tokens with the same slot race.
 *
 * qlin_kv_load_mixed reads slots back as BF16 rows for attention:
 *   k_out, v_out [T, H, D] BF16: RN_bf16(code * scale) (the product is exact
 *   in fp32); a negative slot gives a row of +0; a slot >= num_slots gives +0
 *   and sets the device status word to QLIN_ERR_INVALID_ARG.
 *
 * Both: T == 0 enqueues nothing; all pointers 16-byte aligned device pointers;
 * no workspace.
 */
qlin_status qlin_kv_store_mixed(int64_t T, int64_t H, int64_t D, const void *k, int64_t ldk, const void *v,
                                int64_t ldv, const int64_t *slots, int64_t num_slots, void *k_cache,
                                void *k_scale, void *v_cache, void *v_scale, qlin_stream_t stream);
qlin_status qlin_kv_load_mixed(int64_t T, int64_t H, int64_t D, const int64_t *slots, int64_t num_slots,
                               const void *k_cache, const void *k_scale, const void *v_cache,
                               const void *v_scale, void *k_out, void *v_out, qlin_stream_t stream);

/* Workspace bytes an operation needs for these sizes (0 if none).  Returns
 * (size_t)-1 for invalid arguments. */
size_t qlin_workspace_bytes(qlin_op op, qlin_qtype qtype, int64_t M, int64_t K, int64_t N);

/* Synchronizes `stream`, then reports and clears the device status word of the
 * current device: QLIN_OK, or QLIN_ERR_TIMEOUT if a bounded device-side wait ran
 * out since the last call, QLIN_ERR_INVALID_ARG if a KV-cache kernel met a slot
 * beyond the cache, or QLIN_ERR_CUDA if the stream reported an error.  The
 * first error recorded since the last call wins. */
qlin_status qlin_get_device_status(qlin_stream_t stream);

/* Static, human-readable name of a status code. */
const char *qlin_status_string(qlin_status status);

/* Name of the kernel (or kernel sequence, joined by '+') that the given
 * operation launches for these sizes; "invalid" for arguments it would reject.
 * Pure host function: no device work. */
const char *qlin_kernel_name(qlin_op op, qlin_qtype qtype, int64_t M, int64_t K, int64_t N);

/* Total number of kernels this process has enqueued through the library so far
 * (all devices, all streams; memsets not counted).  Host-side counter. */
uint64_t qlin_launch_count(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int qlin_version(void);

/*
 * Failure-detection check: launches one thread that waits for *flag to become
 * non-zero for at most timeout_ns nanoseconds of GPU global time (capped at
 * 1e9).  If the flag is still zero it sets the device status word to
 * QLIN_ERR_TIMEOUT and returns; it never hangs.  flag is a device pointer.
 */
qlin_status qlin_debug_wait_flag(const uint32_t *flag, uint64_t timeout_ns, qlin_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* QLIN_H_ */
