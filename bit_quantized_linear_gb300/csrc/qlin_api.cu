// C-ABI shim of libqlin: argument validation, workspace sizing, kernel choice
// by shape, and launches on the caller's stream.  No entry point allocates
// device memory or throws; every failure is a qlin_status.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace qlin {

// Device status word (one per device context); set by bounded device waits.
__device__ unsigned g_device_status = 0;

static std::atomic<uint64_t> g_launches{0};
void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

static DeviceInfo g_dev[kMaxDevices];
static std::mutex g_dev_mu;

// SM count of the current device for host-side tile choices that name a
// kernel without launching it: the cached value, else 152 (GB300).
static int sm_count() {
  int d = -1;
  if (cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < kMaxDevices) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev[d].device == d && g_dev[d].sms > 0) return g_dev[d].sms;
  }
  return 152;
}

// Caches the SM count, compute capability and status-word address of the
// current device.  Returns QLIN_OK or an error status.
static qlin_status current_device(DeviceInfo **out) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return QLIN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo &di = g_dev[d];
  if (di.device != d) {
    DeviceInfo t;
    t.device = d;
    if (cudaDeviceGetAttribute(&t.sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.cc_major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.cc_minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess)
      return QLIN_ERR_CUDA;
    if (t.cc_major != 10 || t.cc_minor != 3) return QLIN_ERR_UNSUPPORTED;  // built for sm_103a only
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return QLIN_ERR_CUDA;
    t.status = (unsigned *)p;
    di = t;
  }
  *out = &di;
  return QLIN_OK;
}

// Failure-detection check kernel: waits on a flag with a global-time limit.
__global__ void k_debug_wait(const volatile uint32_t *flag, uint64_t timeout_ns, unsigned *status) {
  pdl_wait();
  pdl_trigger();
  const uint64_t t0 = globaltimer_ns();
  while (*flag == 0u) {
    if (globaltimer_ns() - t0 > timeout_ns) {
      set_status(status, QLIN_ERR_TIMEOUT);
      return;
    }
    __nanosleep(1000);
  }
}

cudaError_t launch_debug_wait(const uint32_t *flag, uint64_t timeout_ns, unsigned *status,
                              cudaStream_t st) {
  return launch_kernel(k_debug_wait, dim3(1), dim3(1), 0, st, 1, (const volatile uint32_t *)flag, timeout_ns, status);
}

static inline bool al16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
static inline bool valid_qtype(int t) { return t == QLIN_INT8 || t == QLIN_E4M3; }
static inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
static inline qlin_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QLIN_OK : QLIN_ERR_CUDA; }

// Common shape checks of the linear entry points.
static qlin_status check_linear_shape(int64_t M, int64_t K, int64_t N) {
  if (M < 0 || K < 16 || N < 16 || (K % 16) || (N % 16)) return QLIN_ERR_INVALID_ARG;
  if (M > (int64_t)1 << 31 || K > (int64_t)1 << 17 || N > (int64_t)1 << 31) return QLIN_ERR_INVALID_ARG;
  return QLIN_OK;
}

// INT8 W8A8 with a static scale and one token tile (M <= 64): the GEMM kernel
// quantizes its activation tiles itself (one kernel, no workspace round trip).
// Larger batches quantize once in a separate pass, which every output tile then
// reuses.
static bool i8_fused_quant(int64_t M) { return M <= 64; }

// Merged gate_up: I output channels (a multiple of 128: both kernels pair whole
// gate and up row blocks), weight rows 2I.
static qlin_status check_glu_shape(int64_t M, int64_t K, int64_t I) {
  if (I < 128 || (I % 128) || I > (int64_t)1 << 30) return QLIN_ERR_INVALID_ARG;
  return check_linear_shape(M, K, 2 * I);
}

// Argument checks of the W8A8 static linear, apart from its workspace (the
// allocation-free entry point makes the same checks in the same order).
qlin_status w8a8_check_args(int qtype, int64_t M, int64_t K, int64_t N, const void *x, const float *input_scale,
                            const void *qw, const float *w_scale, const void *bias, const void *y) {
  if (!valid_qtype(qtype)) return QLIN_ERR_INVALID_ARG;
  if (qlin_status s = check_linear_shape(M, K, N)) return s;
  if (!input_scale || !qw || !w_scale || !al16(qw) || !al16(w_scale) || (bias && !al16(bias)) ||
      ((uintptr_t)input_scale & 3u))
    return QLIN_ERR_INVALID_ARG;
  if (M > 0 && (!x || !y || !al16(x) || !al16(y))) return QLIN_ERR_INVALID_ARG;
  return QLIN_OK;
}

// QLIN_OK when the current device is one the library runs on (sm_103a).
qlin_status device_ready() {
  DeviceInfo *dev;
  return current_device(&dev);
}

}  // namespace qlin

using namespace qlin;

extern "C" {

int qlin_version(void) { return 100; }

uint64_t qlin_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *qlin_kernel_name(qlin_op op, qlin_qtype qtype, int64_t M, int64_t K, int64_t N) {
  if (!valid_qtype(qtype)) return "invalid";
  switch (op) {
    case QLIN_OP_QUANTIZE_WEIGHT: return "k_quantize_weight";
    case QLIN_OP_ACT_SCALE: return "k_absmax_bf16+k_scale_finalize";
    case QLIN_OP_QUANTIZE_ACT: return "k_quantize_act";
    case QLIN_OP_W8A16_GATE_UP_SILU:
      if (check_glu_shape(M, K, N)) return "invalid";
      return qlin_kernel_name(QLIN_OP_W8A16_LINEAR, qtype, M, K, 2 * N);
    case QLIN_OP_W8A8_GATE_UP_SILU:
      if (check_glu_shape(M, K, N)) return "invalid";
      return qlin_kernel_name(QLIN_OP_W8A8_LINEAR, qtype, M, K, 2 * N);
    case QLIN_OP_W8A16_LINEAR: {
      if (check_linear_shape(M, K, N)) return "invalid";
      if (M == 0) return "none";
      if (qtype == QLIN_E4M3 && M <= kW8A16F8MaxM) {
        return w8a16_f8_tt(M) <= 16 ? "k_w8a16_split+k_w8a16_f8<16>" : "k_w8a16_split+k_w8a16_f8<32>";
      }
      static const char *names[5] = {"k_w8_dq<16>", "k_w8_dq<32>", "k_w8_dq<64>", "k_w8_dq<128>", "k_w8_dq<256>"};
      const int b = w8_swap_bnt(M, N, K, sm_count());
      return names[b == 16 ? 0 : b == 32 ? 1 : b == 64 ? 2 : b == 128 ? 3 : 4];
    }
    case QLIN_OP_I8_GEMM_S32: {
      if (check_linear_shape(M, K, N)) return "invalid";
      if (M == 0) return "none";
      static const char *names[4] = {"k_i8_to_bf16+k_w8_dq<16,i8>", "k_i8_to_bf16+k_w8_dq<32,i8>",
                                     "k_i8_to_bf16+k_w8_dq<64,i8>", "k_i8_to_bf16+k_w8_dq<128,i8>"};
      const int b = i8_swap_bnt(M);
      return names[b == 16 ? 0 : b == 32 ? 1 : b == 64 ? 2 : 3];
    }
    case QLIN_OP_W8A8_DYNAMIC_LINEAR: {
      if (check_linear_shape(M, K, N)) return "invalid";
      if (M == 0) return "none";
      if (qtype == QLIN_E4M3) return "k_quantize_act_dyn+k_fp8_gemm";
      static const char *names[4] = {"k_quantize_act_dyn+k_w8_dq<16,i8>", "k_quantize_act_dyn+k_w8_dq<32,i8>",
                                     "k_quantize_act_dyn+k_w8_dq<64,i8>", "k_quantize_act_dyn+k_w8_dq<128,i8>"};
      const int b = i8_swap_bnt(M);
      return names[b == 16 ? 0 : b == 32 ? 1 : b == 64 ? 2 : 3];
    }
    case QLIN_OP_KV_STORE_MIXED:
    case QLIN_OP_KV_LOAD_MIXED: {
      // M = tokens, K = head_dim, N = kv heads
      if (M < 0 || N < 1 || !(K == 32 || K == 64 || K == 128 || K == 256)) return "invalid";
      if (M == 0) return "none";
      static const char *st[4] = {"k_kv_store_mixed<32>", "k_kv_store_mixed<64>", "k_kv_store_mixed<128>",
                                  "k_kv_store_mixed<256>"};
      static const char *ld[4] = {"k_kv_load_mixed<32>", "k_kv_load_mixed<64>", "k_kv_load_mixed<128>",
                                  "k_kv_load_mixed<256>"};
      const int i = K == 32 ? 0 : K == 64 ? 1 : K == 128 ? 2 : 3;
      return op == QLIN_OP_KV_STORE_MIXED ? st[i] : ld[i];
    }
    case QLIN_OP_W8A8_LINEAR: {
      if (check_linear_shape(M, K, N)) return "invalid";
      if (M == 0) return "none";
      if (qtype == QLIN_E4M3) return fp8_xq_used(M, K, N, sm_count()) ? "k_fp8_gemm<xq>" : "k_quantize_act+k_fp8_gemm";
      static const char *names[4] = {"k_quantize_act_i8bf16+k_w8_dq<16,i8>",
                                     "k_quantize_act_i8bf16+k_w8_dq<32,i8>",
                                     "k_quantize_act_i8bf16+k_w8_dq<64,i8>",
                                     "k_quantize_act_i8bf16+k_w8_dq<128,i8>"};
      static const char *fused[4] = {"k_w8_dq<16,i8,xq>", "k_w8_dq<32,i8,xq>", "k_w8_dq<64,i8,xq>", "invalid"};
      const int b = i8_swap_bnt(M);
      return (i8_fused_quant(M) ? fused : names)[b == 16 ? 0 : b == 32 ? 1 : b == 64 ? 2 : 3];
    }
  }
  return "invalid";
}

const char *qlin_status_string(qlin_status s) {
  switch (s) {
    case QLIN_OK: return "QLIN_OK";
    case QLIN_ERR_INVALID_ARG: return "QLIN_ERR_INVALID_ARG";
    case QLIN_ERR_UNSUPPORTED: return "QLIN_ERR_UNSUPPORTED";
    case QLIN_ERR_WORKSPACE: return "QLIN_ERR_WORKSPACE";
    case QLIN_ERR_CUDA: return "QLIN_ERR_CUDA";
    case QLIN_ERR_TIMEOUT: return "QLIN_ERR_TIMEOUT";
  }
  return "QLIN_ERR_UNKNOWN";
}

size_t qlin_workspace_bytes(qlin_op op, qlin_qtype qtype, int64_t M, int64_t K, int64_t N) {
  if (!valid_qtype(qtype) || M < 0 || K < 0 || N < 0) return (size_t)-1;
  switch (op) {
    case QLIN_OP_QUANTIZE_WEIGHT: return 0;
    case QLIN_OP_ACT_SCALE: return 256;
    case QLIN_OP_QUANTIZE_ACT: return 0;
    // E4M3 up to kW8A16F8MaxM tokens: the activations' four E4M3 terms and per-token scales
    case QLIN_OP_W8A16_LINEAR:
    case QLIN_OP_W8A16_GATE_UP_SILU:
      return (qtype == QLIN_E4M3 && M > 0 && M <= kW8A16F8MaxM) ? w8a16_f8_workspace(M, K) : 0;
    // quantized activations: E4M3 codes (1 byte) and, for the fused-quantization GEMM, its
    // task flags; or INT8 codes as integer-valued BF16 (2 bytes)
    case QLIN_OP_W8A8_LINEAR:
    case QLIN_OP_W8A8_GATE_UP_SILU:
      if (qtype == QLIN_E4M3) return round_up((size_t)M * (size_t)K, 256) + round_up(fp8_xq_flag_bytes(M, K), 256);
      return round_up((size_t)M * (size_t)K * 2, 256);
    case QLIN_OP_I8_GEMM_S32: return round_up((size_t)M * (size_t)K * 2, 256);
    // per-token codes (as for the static path) followed by the per-token scales
    case QLIN_OP_W8A8_DYNAMIC_LINEAR:
      return round_up((size_t)M * (size_t)K * (qtype == QLIN_INT8 ? 2 : 1), 256) + round_up((size_t)M * 4, 256);
    case QLIN_OP_KV_STORE_MIXED:
    case QLIN_OP_KV_LOAD_MIXED:
      return 0;
  }
  return (size_t)-1;
}

qlin_status qlin_quantize_weight(qlin_qtype qtype, int64_t N, int64_t K, const float *w, void *qw,
                                 float *w_scale, qlin_stream_t stream) {
  if (!valid_qtype(qtype)) return QLIN_ERR_INVALID_ARG;
  if (N < 0 || K < 16 || (K % 16) || N > ((int64_t)1 << 31) - 1) return QLIN_ERR_INVALID_ARG;
  if (!w || !qw || !w_scale || !al16(w) || !al16(qw) || !al16(w_scale)) return QLIN_ERR_INVALID_ARG;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  return from_cuda(launch_quantize_weight(qtype, N, K, w, qw, w_scale, (cudaStream_t)stream));
}

qlin_status qlin_act_scale_from_calib(qlin_qtype qtype, int64_t rows, int64_t K, const void *x_cal,
                                      float *input_scale, void *ws, size_t ws_bytes,
                                      qlin_stream_t stream) {
  if (!valid_qtype(qtype)) return QLIN_ERR_INVALID_ARG;
  if (rows < 1 || K < 16 || (K % 16)) return QLIN_ERR_INVALID_ARG;
  if (!x_cal || !input_scale || !al16(x_cal) || !al16(input_scale)) return QLIN_ERR_INVALID_ARG;
  if (!ws || !al16(ws) || ws_bytes < qlin_workspace_bytes(QLIN_OP_ACT_SCALE, qtype, rows, K, 0))
    return QLIN_ERR_WORKSPACE;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  return from_cuda(launch_act_scale(qtype, rows, K, x_cal, input_scale, ws, dev->sms,
                                    (cudaStream_t)stream));
}

qlin_status qlin_quantize_act_static(qlin_qtype qtype, int64_t M, int64_t K, const void *x,
                                     const float *input_scale, void *qx, qlin_stream_t stream) {
  if (!valid_qtype(qtype)) return QLIN_ERR_INVALID_ARG;
  if (M < 0 || K < 16 || (K % 16)) return QLIN_ERR_INVALID_ARG;
  if (!input_scale || ((uintptr_t)input_scale & 3u)) return QLIN_ERR_INVALID_ARG;
  if (M > 0 && (!x || !qx || !al16(x) || !al16(qx))) return QLIN_ERR_INVALID_ARG;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (M == 0) return QLIN_OK;
  return from_cuda(launch_quantize_act(qtype, M, K, x, input_scale, qx, dev->sms, (cudaStream_t)stream));
}

qlin_status qlin_w8a16_linear(qlin_qtype qtype, int64_t M, int64_t K, int64_t N, const void *x,
                              const void *qw, const float *w_scale, const void *bias, void *y,
                              void *ws, size_t ws_bytes, qlin_stream_t stream) {
  if (!valid_qtype(qtype)) return QLIN_ERR_INVALID_ARG;
  if (qlin_status s = check_linear_shape(M, K, N)) return s;
  if (!qw || !w_scale || !al16(qw) || !al16(w_scale) || (bias && !al16(bias))) return QLIN_ERR_INVALID_ARG;
  if (M > 0 && (!x || !y || !al16(x) || !al16(y))) return QLIN_ERR_INVALID_ARG;
  const size_t need = qlin_workspace_bytes(QLIN_OP_W8A16_LINEAR, qtype, M, K, N);
  if (need && (!ws || !al16(ws) || ws_bytes < need)) return QLIN_ERR_WORKSPACE;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (M == 0) return QLIN_OK;
  GemmArgs g{kW8A16, qtype, M, K, N, x, qw, w_scale, nullptr, (const uint16_t *)bias, y};
  // E4M3 weights, small batch: FP8 MMAs on the codes against the split activations
  if (qtype == QLIN_E4M3 && M <= kW8A16F8MaxM) return from_cuda(launch_w8a16_f8(g, ws, *dev, (cudaStream_t)stream));
  return from_cuda(launch_w8a16_swap(g, *dev, (cudaStream_t)stream));
}

qlin_status qlin_w8a8_linear(qlin_qtype qtype, int64_t M, int64_t K, int64_t N, const void *x,
                             const float *input_scale, const void *qw, const float *w_scale,
                             const void *bias, void *y, void *ws, size_t ws_bytes,
                             qlin_stream_t stream) {
  if (qlin_status s = w8a8_check_args(qtype, M, K, N, x, input_scale, qw, w_scale, bias, y)) return s;
  const size_t need = qlin_workspace_bytes(QLIN_OP_W8A8_LINEAR, qtype, M, K, N);
  if (need && (!ws || !al16(ws) || ws_bytes < need)) return QLIN_ERR_WORKSPACE;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (M == 0) return QLIN_OK;
  cudaStream_t st = (cudaStream_t)stream;
  GemmArgs g{kW8A8, qtype, M, K, N, ws, qw, w_scale, input_scale, (const uint16_t *)bias, y};
  if (qtype == QLIN_E4M3) {
    if (fp8_xq_used(M, K, g.N, dev->sms)) {  // one kernel: quantization overlapped with the GEMM
      g.xq = x;
      g.xq_flags = (unsigned *)((char *)ws + round_up((size_t)M * (size_t)K, 256));
      return from_cuda(launch_fp8_gemm(g, *dev, st));
    }
    if (launch_quantize_act(qtype, M, K, x, input_scale, ws, dev->sms, st) != cudaSuccess) return QLIN_ERR_CUDA;
    return from_cuda(launch_fp8_gemm(g, *dev, st));
  }
  if (i8_fused_quant(M)) return from_cuda(launch_i8_swap(g, x, false, *dev, st, true));
  if (launch_quantize_act_i8bf16(M, K, x, input_scale, ws, dev->sms, st) != cudaSuccess) return QLIN_ERR_CUDA;
  return from_cuda(launch_i8_swap(g, ws, false, *dev, st));
}

qlin_status qlin_quantize_act_dynamic(qlin_qtype qtype, int64_t M, int64_t K, const void *x, void *qx,
                                      float *x_scale, qlin_stream_t stream) {
  if (!valid_qtype(qtype)) return QLIN_ERR_INVALID_ARG;
  if (M < 0 || K < 16 || (K % 16) || M > ((int64_t)1 << 31) - 1) return QLIN_ERR_INVALID_ARG;
  if (M > 0 && (!x || !qx || !x_scale || !al16(x) || !al16(qx) || !al16(x_scale))) return QLIN_ERR_INVALID_ARG;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (M == 0) return QLIN_OK;
  return from_cuda(launch_quantize_act_dyn(qtype, false, M, K, x, x_scale, qx, (cudaStream_t)stream));
}

qlin_status qlin_w8a8_dynamic_linear(qlin_qtype qtype, int64_t M, int64_t K, int64_t N, const void *x,
                                     const void *qw, const float *w_scale, const void *bias, void *y, void *ws,
                                     size_t ws_bytes, qlin_stream_t stream) {
  if (!valid_qtype(qtype)) return QLIN_ERR_INVALID_ARG;
  if (qlin_status s = check_linear_shape(M, K, N)) return s;
  if (!qw || !w_scale || !al16(qw) || !al16(w_scale) || (bias && !al16(bias))) return QLIN_ERR_INVALID_ARG;
  if (M > 0 && (!x || !y || !al16(x) || !al16(y))) return QLIN_ERR_INVALID_ARG;
  const size_t need = qlin_workspace_bytes(QLIN_OP_W8A8_DYNAMIC_LINEAR, qtype, M, K, N);
  if (need && (!ws || !al16(ws) || ws_bytes < need)) return QLIN_ERR_WORKSPACE;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (M == 0) return QLIN_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const bool i8 = qtype == QLIN_INT8;
  void *codes = ws;
  float *scales = (float *)((char *)ws + round_up((size_t)M * (size_t)K * (i8 ? 2 : 1), 256));
  if (launch_quantize_act_dyn(qtype, i8, M, K, x, scales, codes, st) != cudaSuccess) return QLIN_ERR_CUDA;
  GemmArgs g{kW8A8, qtype, M, K, N, codes, qw, w_scale, scales, (const uint16_t *)bias, y};
  g.x_scale_per_token = 1;
  if (!i8) return from_cuda(launch_fp8_gemm(g, *dev, st));
  return from_cuda(launch_i8_swap(g, codes, false, *dev, st));
}

qlin_status qlin_i8_gemm_s32(int64_t M, int64_t K, int64_t N, const void *qx, const void *qw,
                             int32_t *acc, void *ws, size_t ws_bytes, qlin_stream_t stream) {
  if (qlin_status s = check_linear_shape(M, K, N)) return s;
  if (!qw || !al16(qw)) return QLIN_ERR_INVALID_ARG;
  if (M > 0 && (!qx || !acc || !al16(qx) || !al16(acc))) return QLIN_ERR_INVALID_ARG;
  const size_t need = qlin_workspace_bytes(QLIN_OP_I8_GEMM_S32, QLIN_INT8, M, K, N);
  if (need && (!ws || !al16(ws) || ws_bytes < need)) return QLIN_ERR_WORKSPACE;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (M == 0) return QLIN_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (launch_i8_to_bf16(M, K, qx, ws, dev->sms, st) != cudaSuccess) return QLIN_ERR_CUDA;
  GemmArgs g{kI8Raw, QLIN_INT8, M, K, N, ws, qw, nullptr, nullptr, nullptr, acc};
  return from_cuda(launch_i8_swap(g, ws, true, *dev, st));
}

qlin_status qlin_w8a16_gate_up_silu(qlin_qtype qtype, int64_t M, int64_t K, int64_t I, const void *x,
                                    const void *qw, const float *w_scale, const void *bias, void *y, void *ws,
                                    size_t ws_bytes, qlin_stream_t stream) {
  if (!valid_qtype(qtype)) return QLIN_ERR_INVALID_ARG;
  if (qlin_status s = check_glu_shape(M, K, I)) return s;
  if (!qw || !w_scale || !al16(qw) || !al16(w_scale) || (bias && !al16(bias))) return QLIN_ERR_INVALID_ARG;
  if (M > 0 && (!x || !y || !al16(x) || !al16(y))) return QLIN_ERR_INVALID_ARG;
  const size_t need = qlin_workspace_bytes(QLIN_OP_W8A16_GATE_UP_SILU, qtype, M, K, I);
  if (need && (!ws || !al16(ws) || ws_bytes < need)) return QLIN_ERR_WORKSPACE;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (M == 0) return QLIN_OK;
  GemmArgs g{kW8A16, qtype, M, K, I, x, qw, w_scale, nullptr, (const uint16_t *)bias, y};
  g.glu = 1;
  if (qtype == QLIN_E4M3 && M <= kW8A16F8MaxM) return from_cuda(launch_w8a16_f8(g, ws, *dev, (cudaStream_t)stream));
  return from_cuda(launch_w8a16_swap(g, *dev, (cudaStream_t)stream));
}

qlin_status qlin_w8a8_gate_up_silu(qlin_qtype qtype, int64_t M, int64_t K, int64_t I, const void *x,
                                   const float *input_scale, const void *qw, const float *w_scale,
                                   const void *bias, void *y, void *ws, size_t ws_bytes, qlin_stream_t stream) {
  if (!valid_qtype(qtype)) return QLIN_ERR_INVALID_ARG;
  if (qlin_status s = check_glu_shape(M, K, I)) return s;
  if (!input_scale || !qw || !w_scale || !al16(qw) || !al16(w_scale) || (bias && !al16(bias)) ||
      ((uintptr_t)input_scale & 3u))
    return QLIN_ERR_INVALID_ARG;
  if (M > 0 && (!x || !y || !al16(x) || !al16(y))) return QLIN_ERR_INVALID_ARG;
  const size_t need = qlin_workspace_bytes(QLIN_OP_W8A8_GATE_UP_SILU, qtype, M, K, I);
  if (need && (!ws || !al16(ws) || ws_bytes < need)) return QLIN_ERR_WORKSPACE;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (M == 0) return QLIN_OK;
  cudaStream_t st = (cudaStream_t)stream;
  GemmArgs g{kW8A8, qtype, M, K, I, ws, qw, w_scale, input_scale, (const uint16_t *)bias, y};
  g.glu = 1;
  if (qtype == QLIN_E4M3) {
    if (fp8_xq_used(M, K, 2 * g.N, dev->sms)) {  // one kernel: quantization overlapped with the GEMM
      g.xq = x;
      g.xq_flags = (unsigned *)((char *)ws + round_up((size_t)M * (size_t)K, 256));
      return from_cuda(launch_fp8_gemm(g, *dev, st));
    }
    if (launch_quantize_act(qtype, M, K, x, input_scale, ws, dev->sms, st) != cudaSuccess) return QLIN_ERR_CUDA;
    return from_cuda(launch_fp8_gemm(g, *dev, st));
  }
  if (i8_fused_quant(M)) return from_cuda(launch_i8_swap(g, x, false, *dev, st, true));
  if (launch_quantize_act_i8bf16(M, K, x, input_scale, ws, dev->sms, st) != cudaSuccess) return QLIN_ERR_CUDA;
  return from_cuda(launch_i8_swap(g, ws, false, *dev, st));
}

// Shared argument checks of the two KV-cache entry points.
static qlin_status check_kv(int64_t T, int64_t H, int64_t D, const int64_t *slots, int64_t num_slots,
                            const void *k_cache, const void *k_scale, const void *v_cache, const void *v_scale) {
  if (T < 0 || H < 1 || num_slots < 0) return QLIN_ERR_INVALID_ARG;
  if (!(D == 32 || D == 64 || D == 128 || D == 256)) return QLIN_ERR_INVALID_ARG;
  if (H > 4096 || T > ((int64_t)1 << 40) / H || num_slots > ((int64_t)1 << 40) / H) return QLIN_ERR_INVALID_ARG;
  if (T == 0) return QLIN_OK;
  if (!slots || !al16(slots)) return QLIN_ERR_INVALID_ARG;
  if (!k_cache || !k_scale || !v_cache || !v_scale) return QLIN_ERR_INVALID_ARG;
  if (!al16(k_cache) || !al16(k_scale) || !al16(v_cache) || !al16(v_scale)) return QLIN_ERR_INVALID_ARG;
  return QLIN_OK;
}

qlin_status qlin_kv_store_mixed(int64_t T, int64_t H, int64_t D, const void *k, int64_t ldk, const void *v,
                                int64_t ldv, const int64_t *slots, int64_t num_slots, void *k_cache,
                                void *k_scale, void *v_cache, void *v_scale, qlin_stream_t stream) {
  if (qlin_status s = check_kv(T, H, D, slots, num_slots, k_cache, k_scale, v_cache, v_scale)) return s;
  if (T > 0) {
    if (!k || !v || !al16(k) || !al16(v)) return QLIN_ERR_INVALID_ARG;
    if (ldk < H * D || ldv < H * D || (ldk % 8) || (ldv % 8)) return QLIN_ERR_INVALID_ARG;
  }
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (T == 0) return QLIN_OK;
  KvArgs a{T, H, D, k, v, ldk, ldv, slots, num_slots, k_cache, k_scale, v_cache, v_scale, nullptr, nullptr};
  return from_cuda(launch_kv_store(a, dev->status, dev->sms, (cudaStream_t)stream));
}

qlin_status qlin_kv_load_mixed(int64_t T, int64_t H, int64_t D, const int64_t *slots, int64_t num_slots,
                               const void *k_cache, const void *k_scale, const void *v_cache,
                               const void *v_scale, void *k_out, void *v_out, qlin_stream_t stream) {
  if (qlin_status s = check_kv(T, H, D, slots, num_slots, k_cache, k_scale, v_cache, v_scale)) return s;
  if (T > 0 && (!k_out || !v_out || !al16(k_out) || !al16(v_out))) return QLIN_ERR_INVALID_ARG;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (T == 0) return QLIN_OK;
  KvArgs a{T, H, D, nullptr, nullptr, 0, 0, slots, num_slots, (void *)k_cache, (void *)k_scale,
           (void *)v_cache, (void *)v_scale, k_out, v_out};
  return from_cuda(launch_kv_load(a, dev->status, (cudaStream_t)stream));
}

qlin_status qlin_get_device_status(qlin_stream_t stream) {
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return QLIN_ERR_CUDA;
  unsigned v = 0, zero = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return QLIN_ERR_CUDA;
  if (v && cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return QLIN_ERR_CUDA;
  return v ? (qlin_status)v : QLIN_OK;
}

qlin_status qlin_debug_wait_flag(const uint32_t *flag, uint64_t timeout_ns, qlin_stream_t stream) {
  if (!flag || ((uintptr_t)flag & 3u)) return QLIN_ERR_INVALID_ARG;
  if (timeout_ns > 1000000000ull) timeout_ns = 1000000000ull;
  DeviceInfo *dev;
  if (qlin_status s = current_device(&dev)) return s;
  return from_cuda(launch_debug_wait(flag, timeout_ns, dev->status, (cudaStream_t)stream));
}

}  // extern "C"
