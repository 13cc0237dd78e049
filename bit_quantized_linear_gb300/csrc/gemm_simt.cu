// Plain CUDA-core GEMM for every mode (W8A16, W8A8, raw INT8).  It is the
// simple, obviously-correct kernel the tensor-core paths are checked against
// on the device and the path for shapes the tensor-core kernels do not take.
// Tile 64 (m) x 64 (n) x 32 (k), 256 threads, 4x4 outputs per thread.
// INT8 x INT8 accumulates in int32 (exact); every other mode in fp32 on exact
// operand values.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace qlin {

namespace {
constexpr int BM = 64, BN = 64, BK = 32;

template <int MODE, int QT>
__global__ void __launch_bounds__(256) k_gemm_simt(GemmArgs g) {
  constexpr bool kInt = (MODE != kW8A16) && (QT == QLIN_INT8);
  using Acc = typename std::conditional<kInt, int, float>::type;
  __shared__ Acc As[BK][BM + 1];
  __shared__ Acc Bs[BK][BN + 1];
  const int tid = threadIdx.x;
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
  const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
  Acc acc[4][4] = {};
  for (int64_t k0 = 0; k0 < g.K; k0 += BK) {
    for (int i = tid; i < BM * BK; i += 256) {
      int r = i / BK, c = i % BK;
      int64_t m = m0 + r, k = k0 + c;
      Acc v = 0;
      if (m < g.M && k < g.K) {
        if constexpr (MODE == kW8A16) {
          v = bf16_bits_to_f32(((const uint16_t *)g.a)[m * g.K + k]);
        } else if constexpr (kInt) {
          v = (int)((const int8_t *)g.a)[m * g.K + k];
        } else {
          v = code_to_f32<QT>(((const uint8_t *)g.a)[m * g.K + k]);
        }
      }
      As[c][r] = v;
    }
    for (int i = tid; i < BN * BK; i += 256) {
      int r = i / BK, c = i % BK;
      int64_t n = n0 + r, k = k0 + c;
      Acc v = 0;
      if (n < g.N && k < g.K) {
        uint8_t code = ((const uint8_t *)g.qw)[n * g.K + k];
        if constexpr (kInt)
          v = (int)(int8_t)code;
        else
          v = code_to_f32<QT>(code);
      }
      Bs[c][r] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < BK; ++kk) {
      Acc a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][tm + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tn + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if constexpr (kInt)
            acc[i][j] += a[i] * b[j];
          else
            acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    __syncthreads();
  }
  const float sx = (MODE == kW8A8) ? __ldg(g.x_scale) : 1.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + tm + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tn + j;
      if (n >= g.N) continue;
      if constexpr (MODE == kI8Raw) {
        ((int32_t *)g.y)[m * g.N + n] = (int32_t)acc[i][j];
      } else {
        const float scale = (MODE == kW8A8) ? sx * __ldg(g.w_scale + n) : __ldg(g.w_scale + n);
        const float b = g.bias ? bf16_bits_to_f32(__ldg(g.bias + n)) : 0.0f;
        const float v = fmaf((float)acc[i][j], scale, b);
        ((uint16_t *)g.y)[m * g.N + n] = f32_to_bf16_bits(v);
      }
    }
  }
}
}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs &g, const DeviceInfo &, cudaStream_t st) {
  if (g.M == 0) return cudaSuccess;
  dim3 grid((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM));
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  const bool i8 = g.qtype == QLIN_INT8;
  switch (g.mode) {
    case kW8A16:
      if (i8) k_gemm_simt<kW8A16, QLIN_INT8><<<grid, 256, 0, st>>>(g);
      else k_gemm_simt<kW8A16, QLIN_E4M3><<<grid, 256, 0, st>>>(g);
      break;
    case kW8A8:
      if (i8) k_gemm_simt<kW8A8, QLIN_INT8><<<grid, 256, 0, st>>>(g);
      else k_gemm_simt<kW8A8, QLIN_E4M3><<<grid, 256, 0, st>>>(g);
      break;
    case kI8Raw:
      k_gemm_simt<kI8Raw, QLIN_INT8><<<grid, 256, 0, st>>>(g);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  note_launches(1);
  return cudaGetLastError();
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

}  // namespace qlin
