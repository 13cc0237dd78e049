// Small-batch W8A16 linear on the CUDA cores: y[m, n] = bf16(s_w[n] * sum_k deq(q[n, k]) x[m, k] + b[n])
// for M <= 8 tokens ("Nano-vLLM-MoE" README, "FP8 W8A16 weight-only quantization":
// FP8 weights dequantized to BF16 for a BF16 x BF16 product with fp32
// accumulation; "Nano-vLLM-MOE" README, "INT8 量化支持", the INT8 W8A16 scheme).
//
// At a handful of tokens the layer is a matrix-vector product bound by the
// weight stream (one byte per code, 2M flops per byte): it needs HBM bandwidth,
// not tensor cores.  Each warp takes pairs of weight rows (rows 2g and 2g + 1,
// or gate row g and up row I + g of a merged gate_up weight) and a contiguous
// range of K.  A lane streams 16 codes of each row per step with asynchronous
// 16-byte copies (L2 only) into its own slots of a shared-memory ring, eight
// steps ahead across row pairs, so the weight stream never waits on the
// arithmetic; it reads back only what it copied itself, so no barrier is
// needed.  The codes become exact fp32 values and are accumulated against the
// tokens' BF16 activations (read through L1, shared by every warp) with packed
// f32x2 FMAs.  When there are too few row pairs to occupy every warp, K is
// split over 2 or 4 warps of a CTA and their partial sums meet in shared
// memory.  The first steps' copies are issued before
// waiting for the previous kernel of the stream (programmatic dependent
// launch): the weights do not depend on that kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace qlin {
namespace {

constexpr int kGemvWarps = 8, kGemvThreads = 32 * kGemvWarps;
constexpr int kGemvChunk = 512;  // codes of one row per warp step (16 per lane)
constexpr int kGemvDepth = 8;    // warp steps in flight (ring slots per lane)
// dynamic shared memory: per warp, per step slot, per row of the pair, 32 lanes x 16 bytes
constexpr int kGemvRingBytes = kGemvWarps * kGemvDepth * 2 * 32 * 16;

struct GemvParams {
  int M, N, K;  // N: output channels (I for the merged gate_up)
  int glu;      // merged gate_up: rows g and N + g, y = silu(gate) * up
  int splits;   // warps of a CTA that share one row pair (1, 2 or 4), each a range of K
  int groups;   // row pairs: N / 2, or N for glu
  const uint8_t *qw;
  const float *w_scale;
  const uint16_t *x;
  const uint16_t *bias;
  uint16_t *y;
};

// 16 bytes global -> shared, asynchronous, cached in L2 only; completion per
// thread through commit groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float lo_f(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// 16 codes (one 16-byte word) -> 8 pairs of exact fp32 values, pair i = codes 2i, 2i + 1.
template <int QT>
__device__ __forceinline__ void codes16_to_f32x2(uint4 v, uint64_t (&w)[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  if constexpr (QT == QLIN_INT8) {
    // byte b (two's complement) as 2^23 + (b ^ 0x80) in fp32, minus 2^23 + 128: exact
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t s = u[j] ^ 0x80808080u;
      const uint64_t lo = pack2(__uint_as_float(__byte_perm(s, 0x4B000000u, 0x7540)),
                                __uint_as_float(__byte_perm(s, 0x4B000000u, 0x7541)));
      const uint64_t hi = pack2(__uint_as_float(__byte_perm(s, 0x4B000000u, 0x7542)),
                                __uint_as_float(__byte_perm(s, 0x4B000000u, 0x7543)));
      const uint64_t off = pack2(-8388736.0f, -8388736.0f);
      w[2 * j] = f32x2_add(lo, off);
      w[2 * j + 1] = f32x2_add(hi, off);
    }
  } else {
    // E4M3 pairs -> f16x2 (exact: every E4M3 value is a float16) -> fp32
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const __half2_raw r =
            __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(u[j] >> (16 * h)), __NV_E4M3);
        const float2 f = __half22float2(__half2(r));
        w[2 * j + h] = pack2(f.x, f.y);
      }
    }
  }
}

template <int QT, int MT>
__global__ void __launch_bounds__(kGemvThreads, 2) k_w8_gemv(GemvParams p) {
  __shared__ float red[kGemvWarps][2][MT];  // partial sums of split-K warps
  extern __shared__ __align__(16) uint8_t ring[];  // kGemvRingBytes (lane-contiguous reads)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.splits, slot = warp / S, part = warp % S, slots = kGemvWarps / S;
  const int K = p.K, nch = (K + kGemvChunk - 1) / kGemvChunk;
  const int c0 = part * nch / S, c1 = (part + 1) * nch / S, nc = c1 - c0;  // this warp's chunks of K
  const int stride = gridDim.x * slots, first = blockIdx.x * slots;
  const int rounds = first < p.groups ? (p.groups - first + stride - 1) / stride : 0;  // same for the CTA
  auto rows_of = [&](int g, int &r0, int &r1) {
    r0 = p.glu ? g : 2 * g;
    r1 = p.glu ? p.N + g : 2 * g + 1;
  };
  // step t = chunk c0 + t % nc of the row pair of round t / nc; its copies go to slot t % depth
  const uint32_t ring0 = tc::smem_u32(ring + warp * (kGemvDepth * 2 * 512) + 16 * lane);
  auto issue = [&](int t) {
    if (t < rounds * nc) {
      const int g = first + (t / nc) * stride + slot, k = (c0 + t % nc) * kGemvChunk + 16 * lane;
      if (g < p.groups && k < K) {
        int r0, r1;
        rows_of(g, r0, r1);
        const uint32_t d = ring0 + (uint32_t)((t % kGemvDepth) * 2 * 512);
        cp_async16(d, p.qw + (size_t)r0 * K + k);
        cp_async16(d + 512, p.qw + (size_t)r1 * K + k);
      }
    }
    cp_async_commit();  // one group per step, empty or not: the wait counts stay exact
  };
  // the weights do not depend on the previous kernel of the stream: the first
  // steps are in flight while it finishes
#pragma unroll 1
  for (int t = 0; t < kGemvDepth; ++t) issue(t);
  pdl_wait();  // x and y may belong to the previous kernel from here on
  pdl_trigger();

  for (int r = 0; r < rounds; ++r) {
    const int g = first + r * stride + slot;
    uint64_t acc[2][MT];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[i][m] = 0;
#pragma unroll 1
    for (int cc = 0; cc < nc; ++cc) {
      const int t = r * nc + cc, k = (c0 + cc) * kGemvChunk + 16 * lane;
      cp_async_wait<kGemvDepth - 1>();  // this lane's copies of step t have landed
      const uint32_t d = ring0 + (uint32_t)((t % kGemvDepth) * 2 * 512);
      uint4 va = make_uint4(0, 0, 0, 0), vb = va;
      const bool live = g < p.groups && k < K;
      if (live) va = lds_v4(d), vb = lds_v4(d + 512);
      issue(t + kGemvDepth);  // refills this slot: the reads above are done (same thread)
      if (live) {
        uint64_t fa[8], fb[8];
        codes16_to_f32x2<QT>(va, fa);
        codes16_to_f32x2<QT>(vb, fb);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < p.M) {
            const uint4 *xp = reinterpret_cast<const uint4 *>(p.x + (size_t)m * K + k);
            const uint4 x0 = __ldg(xp), x1 = __ldg(xp + 1);
            const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint64_t xf = pack2(__uint_as_float(xw[q] << 16), __uint_as_float(xw[q] & 0xFFFF0000u));
              acc[0][m] = f32x2_fma(fa[q], xf, acc[0][m]);
              acc[1][m] = f32x2_fma(fb[q], xf, acc[1][m]);
            }
          }
        }
      }
    }
    // lane sums -> warp sums (every lane ends with all of them)
    float s[2][MT];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float v = lo_f(acc[i][m]) + hi_f(acc[i][m]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        s[i][m] = v;
      }
    if (S > 1) {  // the split-K warps of a slot meet in shared memory
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int m = 0; m < MT; ++m) red[warp][i][m] = s[i][m];
      }
      __syncthreads();
      if (part == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            float v = 0.0f;
            for (int w = 0; w < S; ++w) v += red[warp + w][i][m];  // fixed order: deterministic
            s[i][m] = v;
          }
      }
      __syncthreads();  // red is rewritten next round
    }
    if (part == 0 && g < p.groups && lane < MT && lane < p.M) {
      int r0, r1;
      rows_of(g, r0, r1);
      const int m = lane;
      float a0 = s[0][0], a1 = s[1][0];
#pragma unroll
      for (int mm = 1; mm < MT; ++mm)
        if (mm == m) a0 = s[0][mm], a1 = s[1][mm];
      const float y0 = fmaf(a0, __ldg(p.w_scale + r0), p.bias ? bf16_bits_to_f32(__ldg(p.bias + r0)) : 0.0f);
      const float y1 = fmaf(a1, __ldg(p.w_scale + r1), p.bias ? bf16_bits_to_f32(__ldg(p.bias + r1)) : 0.0f);
      if (p.glu) {
        p.y[(size_t)m * p.N + g] = f32_to_bf16_bits(silu_f(y0) * y1);
      } else {
        const uint32_t o = (uint32_t)f32_to_bf16_bits(y0) | ((uint32_t)f32_to_bf16_bits(y1) << 16);
        *reinterpret_cast<uint32_t *>(p.y + (size_t)m * p.N + r0) = o;  // columns 2g, 2g + 1
      }
    }
  }
  cp_async_wait<0>();  // no copy lands after the CTA has left
}

template <int QT, int MT>
cudaError_t launch_gemv_t(const GemvParams &p, int sms, cudaStream_t st) {
  const int slots = kGemvWarps / p.splits;
  int grid = (p.groups + slots - 1) / slots;
  if (grid > 2 * sms) grid = 2 * sms;
  static const cudaError_t attr =
      cudaFuncSetAttribute(k_w8_gemv<QT, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvRingBytes);
  if (attr != cudaSuccess) return attr;
  return launch_kernel(k_w8_gemv<QT, MT>, dim3((unsigned)grid), dim3(kGemvThreads), kGemvRingBytes, st, 1, p);
}

template <int QT>
cudaError_t launch_gemv_q(const GemvParams &p, int sms, cudaStream_t st) {
  if (p.M <= 1) return launch_gemv_t<QT, 1>(p, sms, st);
  if (p.M <= 2) return launch_gemv_t<QT, 2>(p, sms, st);
  if (p.M <= 4) return launch_gemv_t<QT, 4>(p, sms, st);
  return launch_gemv_t<QT, 8>(p, sms, st);
}

}  // namespace

// Split of K over the warps of a CTA: the fewest (1, 2, 4) that give every
// warp on the GPU a row pair at least once.
int w8_gemv_splits(int64_t N, int glu, int sms) {
  const int64_t groups = glu ? N : N / 2, warps = (int64_t)2 * sms * kGemvWarps;
  int s = 1;
  while (s < 4 && groups * s < warps) s *= 2;
  return s;
}

cudaError_t launch_w8_gemv(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st) {
  if (g.M == 0) return cudaSuccess;
  if (g.M > kW8GemvMaxM) return cudaErrorInvalidValue;
  GemvParams p;
  p.M = (int)g.M;
  p.N = (int)g.N;
  p.K = (int)g.K;
  p.glu = g.glu;
  p.splits = w8_gemv_splits(g.N, g.glu, dev.sms);
  p.groups = g.glu ? (int)g.N : (int)(g.N / 2);
  p.qw = (const uint8_t *)g.qw;
  p.w_scale = g.w_scale;
  p.x = (const uint16_t *)g.a;
  p.bias = g.bias;
  p.y = (uint16_t *)g.y;
  return g.qtype == QLIN_INT8 ? launch_gemv_q<QLIN_INT8>(p, dev.sms, st) : launch_gemv_q<QLIN_E4M3>(p, dev.sms, st);
}

}  // namespace qlin
