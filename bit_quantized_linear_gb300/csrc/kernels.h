// Internal launcher declarations shared by the C-ABI shim and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "qlin.h"

namespace qlin {

struct DeviceInfo {
  int device = -1;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
  unsigned *status = nullptr;  // device status word (QLIN_ERR_TIMEOUT on a run-out wait)
};

// Host-side count of kernels enqueued by the library (qlin_launch_count).
void note_launches(int n);

// Argument checks of the W8A8 static linear apart from its workspace, and the
// current-device check (qlin_api.cu); QLIN_OK or the status to return.
qlin_status w8a8_check_args(int qtype, int64_t M, int64_t K, int64_t N, const void *x, const float *input_scale,
                            const void *qw, const float *w_scale, const void *bias, const void *y);
qlin_status device_ready();

// Launches `kernel` on `st` with programmatic stream serialization (the kernel
// calls pdl_wait() before reading global inputs) and an optional cluster
// shape along z.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          unsigned cluster_z, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster_z > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = cluster_z;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// A cooperative launch (every CTA resident at once, which the fused-quantization
// GEMM's cross-CTA flags rely on), with an optional cluster shape along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_coop(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                               unsigned cluster_x, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeCooperative;
  attrs[na].val.cooperative = 1;
  ++na;
  if (cluster_x > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = cluster_x;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e == cudaSuccess) note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// As launch_kernel, with a cluster shape along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_x(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            unsigned cluster_x, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = cluster_x;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// How many clusters of `cz` CTAs along z (block, dynamic shared memory as
// given) can be resident on the current device at once; 0 if the query fails.
// Remembered per device and cluster size in `cache` (kMaxDevices x 9 entries,
// one table per kernel), since the answer depends only on the kernel's
// resources and the device.
constexpr int kMaxDevices = 64;  // devices a process may use (per-device tables)
template <typename... KArgs>
int max_active_clusters_z(void (*kernel)(KArgs...), dim3 block, size_t smem, unsigned cz, int device,
                          std::atomic<int> *cache) {
  if (cz < 2 || cz > 8 || device < 0 || device >= kMaxDevices) return 0;
  std::atomic<int> &slot = cache[device * 9 + cz];
  int n = slot.load(std::memory_order_relaxed);
  if (n > 0) return n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, cz);
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeClusterDimension;
  a.val.clusterDim.x = 1;
  a.val.clusterDim.y = 1;
  a.val.clusterDim.z = cz;
  cfg.attrs = &a;
  cfg.numAttrs = 1;
  n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (const void *)kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  slot.store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t launch_quantize_weight(int qtype, int64_t N, int64_t K, const float *w, void *qw,
                                   float *s, cudaStream_t st);
cudaError_t launch_act_scale(int qtype, int64_t rows, int64_t K, const void *x, float *scale,
                             void *ws, int sms, cudaStream_t st);
cudaError_t launch_quantize_act(int qtype, int64_t M, int64_t K, const void *x, const float *s,
                                void *qx, int sms, cudaStream_t st);

// GEMM epilogue / operand modes.
enum GemmMode {
  kW8A16 = 0,   // A = BF16 x, B = 8-bit weight codes, acc fp32, y = acc*s_w[n] + b
  kW8A8 = 1,    // A = 8-bit activation codes, B = 8-bit weight codes, y = acc*(s_x*s_w[n]) + b
  kI8Raw = 2    // INT8 codes, raw int32 accumulator out
};

struct GemmArgs {
  int mode;
  int qtype;
  int64_t M, K, N;
  const void *a;          // x (BF16) or qx (codes)
  const void *qw;         // [N,K] codes
  const float *w_scale;   // [N]
  const float *x_scale;   // device scalar (kW8A8), per-token [M] (x_scale_per_token), or null
  const uint16_t *bias;   // [N] or null
  void *y;                // [M,N] BF16, or int32 for kI8Raw
  int x_scale_per_token = 0;  // x_scale holds one scale per token row (dynamic W8A8)
  int glu = 0;  // merged gate_up: qw/w_scale/bias have 2N rows (gate rows first), y = silu(gate) * up [M, N]
  // FP8 W8A8 with the static quantization inside the GEMM: `a` is the codes
  // workspace, xq the BF16 activations, xq_flags the zeroed task flags
  const void *xq = nullptr;
  unsigned *xq_flags = nullptr;
};

// E4M3 W8A16 on the FP8 tensor cores (w8a16_f8.cu): up to kW8A16F8MaxM tokens,
// plain or merged gate_up; the activations are split into four E4M3 terms in
// the workspace (w8a16_f8_workspace bytes).
constexpr int kW8A16F8MaxM = 32;
int w8a16_f8_tt(int64_t M);
int w8a16_f8_splits(int units, int kblocks, int sms);
size_t w8a16_f8_workspace(int64_t M, int64_t K);
cudaError_t launch_w8a16_f8(const GemmArgs &g, void *ws, const DeviceInfo &dev, cudaStream_t st);

// Fused-quantization FP8 GEMM: task-flag area (u32) for these sizes, and
// whether the fused kernel is used.
size_t fp8_xq_flag_bytes(int64_t M, int64_t K);
bool fp8_xq_used(int64_t M, int64_t K, int64_t N, int sms);

// Mixed KV cache (kv_kernels.cu): INT8 keys with float16 group-32 scales,
// E4M3 values with float16 per-(token, head) scales.
struct KvArgs {
  int64_t T, H, D;        // tokens, kv heads, head_dim (32, 64, 128 or 256)
  const void *k, *v;      // BF16 rows of the new tokens (store), row strides ldk / ldv elements
  int64_t ldk, ldv;
  const int64_t *slots;   // [T] cache slot of each token; negative = padding
  int64_t num_slots;
  void *k_cache, *k_scale, *v_cache, *v_scale;  // [S,H,D] int8, [S,H,D/32] f16, [S,H,D] e4m3, [S,H] f16
  void *k_out, *v_out;    // BF16 [T,H,D] (load)
};
cudaError_t launch_kv_store(const KvArgs &a, unsigned *status, int sms, cudaStream_t st);
cudaError_t launch_kv_load(const KvArgs &a, unsigned *status, cudaStream_t st);

// tcgen05 kernels (gemm_tc.cu)
cudaError_t launch_fp8_gemm(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st);
cudaError_t launch_w8a16_swap(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st);
cudaError_t launch_i8_swap(const GemmArgs &g, const void *xb, bool raw, const DeviceInfo &dev, cudaStream_t st,
                           bool fused = false);
int w8_swap_bnt(int64_t M, int64_t N, int64_t K, int sms);
int i8_swap_bnt(int64_t M);
int w8_swap_splits(int64_t tiles, int64_t K, int sms, int bnt);

// INT8 operand preparation for the tensor-core INT8 path (quant_kernels.cu)
cudaError_t launch_quantize_act_i8bf16(int64_t M, int64_t K, const void *x, const float *s, void *out, int sms,
                                       cudaStream_t st);
cudaError_t launch_i8_to_bf16(int64_t M, int64_t K, const void *q, void *out, int sms, cudaStream_t st);
// Dynamic per-token quantization: scales s[M]; codes (1 byte) or INT8 codes as BF16.
cudaError_t launch_quantize_act_dyn(int qtype, bool out_bf16, int64_t M, int64_t K, const void *x, float *s, void *q,
                                    cudaStream_t st);

}  // namespace qlin
