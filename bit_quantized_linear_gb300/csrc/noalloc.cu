// qlin_w8a8_linear_noalloc: the W8A8 static linear for callers that cannot
// allocate device memory.  Its scratch (the quantized activations) lives in a
// file-scope device array owned by the library instead of a caller workspace.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace qlin {

// Scratch of the allocation-free W8A8 entry point.  A file-scope device array:
// every GPU that loads the library holds it until the process exits.  All calls
// on a device share it.  A call reads only what it wrote itself: the codes it
// quantized, and the fused FP8 GEMM's task flags, which the call clears on its
// stream before the GEMM starts.
static __device__ __align__(256) uint8_t g_w8a8_scratch[QLIN_W8A8_NOALLOC_SCRATCH_BYTES];

// Host code cannot pass the array's name to a kernel (on the host it is only a
// stand-in symbol), so its device address is looked up once per device with
// cudaGetSymbolAddress while that device is current, and cached here.
static constexpr int kNoallocMaxDevices = 64;
static void *g_scratch_addr[kNoallocMaxDevices];
static std::mutex g_scratch_mu;

static qlin_status scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) return QLIN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_w8a8_scratch) != cudaSuccess || p == nullptr) return QLIN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return QLIN_OK;
}

}  // namespace qlin

extern "C" qlin_status qlin_w8a8_linear_noalloc(qlin_qtype qtype, int64_t M, int64_t K, int64_t N,
                                                const void *x, const float *input_scale, const void *qw,
                                                const float *w_scale, const void *bias, void *y,
                                                qlin_stream_t stream) {
  // the checks of qlin_w8a8_linear in its order: arguments, size, device
  if (qlin_status s = qlin::w8a8_check_args(qtype, M, K, N, x, input_scale, qw, w_scale, bias, y)) return s;
  if (qlin_workspace_bytes(QLIN_OP_W8A8_LINEAR, qtype, M, K, N) > QLIN_W8A8_NOALLOC_SCRATCH_BYTES)
    return QLIN_ERR_WORKSPACE;
  if (qlin_status s = qlin::device_ready()) return s;
  if (M == 0) return QLIN_OK;
  void *scratch = nullptr;
  if (qlin_status s = qlin::scratch_address(&scratch)) return s;
  return qlin_w8a8_linear(qtype, M, K, N, x, input_scale, qw, w_scale, bias, y, scratch,
                          QLIN_W8A8_NOALLOC_SCRATCH_BYTES, stream);
}
