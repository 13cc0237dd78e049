// Quantizers: per-output-channel weight quantization, calibration abs-max and
// static per-tensor activation quantization.  All HBM-streaming kernels with
// 16-byte vector accesses; the arithmetic of one element is qlin::quantize_one
// (the quotient by the scale correctly rounded, then the code).
#include "common.cuh"
#include "kernels.h"

namespace qlin {

// ---------------------------------------------------------------------------
// Weight quantization: one CTA per output row n.
//   pass 1: s = max_k |w[n,k]| / QMAX (s = 1 for an all-zero row)
//   pass 2: q[n,k] = Q(w[n,k] / s), 16 codes (one 16-byte store) per step.
// The second pass re-reads the row, which is at most 76 KB and served by L2.
// ---------------------------------------------------------------------------
template <int QT>
__global__ void __launch_bounds__(256) k_quantize_weight(const float *__restrict__ w,
                                                         uint8_t *__restrict__ q,
                                                         float *__restrict__ s, int64_t K) {
  // No early start of the next kernel: the linears read their weight codes
  // before they wait for their predecessor, so the kernel that writes codes
  // must have completed before any kernel after it begins.
  pdl_wait();
  __shared__ float red[8];
  const int64_t n = blockIdx.x;
  const float4 *row = reinterpret_cast<const float4 *>(w + n * K);
  const int64_t K16 = K / 16;
  float amax = 0.0f;
  for (int64_t i = threadIdx.x; i < K / 4; i += blockDim.x) {
    float4 v = __ldg(row + i);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
  const float sc = amax > 0.0f ? __fdiv_rn(amax, qmax_of(QT)) : 1.0f;
  if (threadIdx.x == 0) s[n] = sc;
  const Scale scl = make_scale(sc);
  uint4 *qrow = reinterpret_cast<uint4 *>(q + n * K);
  for (int64_t i = threadIdx.x; i < K16; i += blockDim.x) {
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float4 v = __ldg(row + 4 * i + j);
      out[j] = (uint32_t)quantize_one<QT, true>(v.x, scl) | ((uint32_t)quantize_one<QT, true>(v.y, scl) << 8) |
               ((uint32_t)quantize_one<QT, true>(v.z, scl) << 16) |
               ((uint32_t)quantize_one<QT, true>(v.w, scl) << 24);
    }
    qrow[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// ---------------------------------------------------------------------------
// Calibration abs-max: grid-stride over 8-element BF16 chunks, CTA reduction,
// then one atomicMax on the fp32 bit pattern (non-negative floats order like
// their bit patterns).  The finalize kernel turns it into the scale.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_absmax_bf16(const uint4 *__restrict__ x, int64_t n8,
                                                     unsigned *__restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8];
  float amax = 0.0f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint4 v = __ldg(x + i);
    uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // |bf16| for both halves: clear the sign bits, then compare as floats.
      amax = fmaxf(amax, __uint_as_float((wds[j] & 0x7FFFu) << 16));
      amax = fmaxf(amax, __uint_as_float(wds[j] & 0x7FFF0000u));
    }
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
    amax = fmaxf(amax, red[0]);
    atomicMax(out, __float_as_uint(amax));
  }
}

__global__ void k_scale_finalize(const unsigned *__restrict__ amax_bits, float *__restrict__ scale,
                                 float qmax) {
  pdl_wait();
  pdl_trigger();
  const float a = __uint_as_float(*amax_bits);
  *scale = a > 0.0f ? __fdiv_rn(a, qmax) : 1.0f;
}

// ---------------------------------------------------------------------------
// Static activation quantization: 16 BF16 in (two 16-byte loads), 16 codes out
// (one 16-byte store) per thread step.  The scale is read from device memory.
// E4M3 on the fast scale range takes the packed form of the same arithmetic.
// ---------------------------------------------------------------------------
template <int QT>
__global__ void __launch_bounds__(256) k_quantize_act(const uint4 *__restrict__ x,
                                                      const float *__restrict__ s_ptr,
                                                      uint4 *__restrict__ q, int64_t n16) {
  pdl_wait();
  pdl_trigger();
  const float sv = __ldg(s_ptr);
  const Scale s = make_scale(sv);
  if constexpr (QT == QLIN_E4M3) {
    if (s.fast) {
      const StaticE4m3 se = make_static_e4m3(sv);
      for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
           i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 a = __ldg(x + 2 * i), b = __ldg(x + 2 * i + 1);
        q[i] = make_uint4(e4m3_static4_fast(a.x, a.y, se), e4m3_static4_fast(a.z, a.w, se),
                          e4m3_static4_fast(b.x, b.y, se), e4m3_static4_fast(b.z, b.w, se));
      }
      return;
    }
  }
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint4 a = __ldg(x + 2 * i), b = __ldg(x + 2 * i + 1);
    uint32_t in[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t lo = in[2 * j], hi = in[2 * j + 1];
      out[j] = (uint32_t)quantize_one<QT, false>(bf16_bits_to_f32(lo & 0xFFFFu), s) |
               ((uint32_t)quantize_one<QT, false>(bf16_bits_to_f32(lo >> 16), s) << 8) |
               ((uint32_t)quantize_one<QT, false>(bf16_bits_to_f32(hi & 0xFFFFu), s) << 16) |
               ((uint32_t)quantize_one<QT, false>(bf16_bits_to_f32(hi >> 16), s) << 24);
    }
    q[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// ---------------------------------------------------------------------------
// INT8 activation codes written as integer-valued BF16 (exact for |q| <= 127):
// the B operand of the INT8 tensor-core path.  8 BF16 in, 8 BF16 codes out.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_quantize_act_i8bf16(const uint4 *__restrict__ x,
                                                            const float *__restrict__ s_ptr,
                                                            uint4 *__restrict__ q, int64_t n8) {
  pdl_wait();
  pdl_trigger();
  const Scale s = make_scale(__ldg(s_ptr));
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 a = __ldg(x + i);
    uint32_t in[4] = {a.x, a.y, a.z, a.w}, out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = (float)(int8_t)quantize_one<QLIN_INT8, false>(bf16_bits_to_f32(in[j] & 0xFFFFu), s);
      const float hi = (float)(int8_t)quantize_one<QLIN_INT8, false>(bf16_bits_to_f32(in[j] >> 16), s);
      out[j] = pack_code_bf16x2(lo, hi);
    }
    q[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// INT8 codes -> integer-valued BF16 (exact).  16 codes in, 16 BF16 out.
__global__ void __launch_bounds__(256) k_i8_to_bf16(const uint4 *__restrict__ q, uint4 *__restrict__ out,
                                                   int64_t n16) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 a = __ldg(q + i);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float lo = (float)(int8_t)(w[j] >> (16 * h));
        const float hi = (float)(int8_t)(w[j] >> (16 * h + 8));
        o[2 * j + h] = pack_code_bf16x2(lo, hi);
      }
    }
    out[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
    out[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// ---------------------------------------------------------------------------
// Dynamic per-token activation quantization: one CTA per token row.
//   pass 1: s[m] = max_k |x[m,k]| / QMAX (1 for an all-zero row)
//   pass 2: codes Q(x / s[m]); OUT_BF16 writes INT8 codes as integer-valued BF16
//           (the operand of the INT8 tensor-core path), else 1-byte codes.
// The second pass re-reads the row (at most 38 KB) from L1/L2.
// ---------------------------------------------------------------------------
template <int QT, bool OUT_BF16>
__global__ void __launch_bounds__(256) k_quantize_act_dyn(const uint16_t *__restrict__ x, float *__restrict__ s_out,
                                                          void *__restrict__ q, int64_t K) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8];
  const int64_t m = blockIdx.x;
  const uint4 *row = reinterpret_cast<const uint4 *>(x + m * K);
  const int64_t K8 = K / 8;
  float amax = 0.0f;
  for (int64_t i = threadIdx.x; i < K8; i += blockDim.x) {
    const uint4 v = __ldg(row + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, __uint_as_float((w[j] & 0x7FFFu) << 16));
      amax = fmaxf(amax, __uint_as_float(w[j] & 0x7FFF0000u));
    }
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
  const float sc = amax > 0.0f ? __fdiv_rn(amax, qmax_of(QT)) : 1.0f;
  if (threadIdx.x == 0) s_out[m] = sc;
  const Scale scl = make_scale(sc);
  for (int64_t i = threadIdx.x; i < K8; i += blockDim.x) {
    const uint4 v = __ldg(row + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (OUT_BF16) {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = (float)(int8_t)quantize_one<QLIN_INT8, true>(bf16_bits_to_f32(w[j] & 0xFFFFu), scl);
        const float hi = (float)(int8_t)quantize_one<QLIN_INT8, true>(bf16_bits_to_f32(w[j] >> 16), scl);
        o[j] = pack_code_bf16x2(lo, hi);
      }
      reinterpret_cast<uint4 *>((uint16_t *)q + m * K)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      uint32_t o[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t lo = w[2 * j], hi = w[2 * j + 1];
        o[j] = (uint32_t)quantize_one<QT, true>(bf16_bits_to_f32(lo & 0xFFFFu), scl) |
               ((uint32_t)quantize_one<QT, true>(bf16_bits_to_f32(lo >> 16), scl) << 8) |
               ((uint32_t)quantize_one<QT, true>(bf16_bits_to_f32(hi & 0xFFFFu), scl) << 16) |
               ((uint32_t)quantize_one<QT, true>(bf16_bits_to_f32(hi >> 16), scl) << 24);
      }
      reinterpret_cast<uint2 *>((uint8_t *)q + m * K)[i] = make_uint2(o[0], o[1]);
    }
  }
}

// --------------------------------- launchers --------------------------------
static int stream_grid(int64_t work, int per_cta, int sms) {
  int64_t g = (work + per_cta - 1) / per_cta;
  int64_t cap = (int64_t)sms * 8;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_quantize_weight(int qtype, int64_t N, int64_t K, const float *w, void *qw,
                                   float *s, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  dim3 grid((unsigned)N), block(256);
  return qtype == QLIN_INT8
             ? launch_kernel(k_quantize_weight<QLIN_INT8>, grid, block, 0, st, 1, w, (uint8_t *)qw, s, K)
             : launch_kernel(k_quantize_weight<QLIN_E4M3>, grid, block, 0, st, 1, w, (uint8_t *)qw, s, K);
}

cudaError_t launch_act_scale(int qtype, int64_t rows, int64_t K, const void *x, float *scale,
                             void *ws, int sms, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  const int64_t n8 = rows * K / 8;
  e = launch_kernel(k_absmax_bf16, dim3(stream_grid(n8, 256 * 4, sms)), dim3(256), 0, st, 1, (const uint4 *)x, n8,
                    (unsigned *)ws);
  if (e != cudaSuccess) return e;
  return launch_kernel(k_scale_finalize, dim3(1), dim3(1), 0, st, 1, (const unsigned *)ws, scale, qmax_of(qtype));
}

cudaError_t launch_quantize_act(int qtype, int64_t M, int64_t K, const void *x, const float *s,
                                void *qx, int sms, cudaStream_t st) {
  const int64_t n16 = M * K / 16;
  if (n16 == 0) return cudaSuccess;
  const int grid = stream_grid(n16, 256, sms);
  return qtype == QLIN_INT8
             ? launch_kernel(k_quantize_act<QLIN_INT8>, dim3(grid), dim3(256), 0, st, 1, (const uint4 *)x, s,
                             (uint4 *)qx, n16)
             : launch_kernel(k_quantize_act<QLIN_E4M3>, dim3(grid), dim3(256), 0, st, 1, (const uint4 *)x, s,
                             (uint4 *)qx, n16);
}

}  // namespace qlin

namespace qlin {
cudaError_t launch_quantize_act_i8bf16(int64_t M, int64_t K, const void *x, const float *s, void *out, int sms,
                                       cudaStream_t st) {
  const int64_t n8 = M * K / 8;
  if (n8 == 0) return cudaSuccess;
  return launch_kernel(k_quantize_act_i8bf16, dim3(stream_grid(n8, 256, sms)), dim3(256), 0, st, 1,
                       (const uint4 *)x, s, (uint4 *)out, n8);
}

cudaError_t launch_i8_to_bf16(int64_t M, int64_t K, const void *q, void *out, int sms, cudaStream_t st) {
  const int64_t n16 = M * K / 16;
  if (n16 == 0) return cudaSuccess;
  return launch_kernel(k_i8_to_bf16, dim3(stream_grid(n16, 256, sms)), dim3(256), 0, st, 1, (const uint4 *)q,
                       (uint4 *)out, n16);
}
}  // namespace qlin

namespace qlin {
cudaError_t launch_quantize_act_dyn(int qtype, bool out_bf16, int64_t M, int64_t K, const void *x, float *s, void *q,
                                    cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const dim3 grid((unsigned)M), block(256);
  if (out_bf16)
    return launch_kernel(k_quantize_act_dyn<QLIN_INT8, true>, grid, block, 0, st, 1, (const uint16_t *)x, s, q, K);
  return qtype == QLIN_INT8
             ? launch_kernel(k_quantize_act_dyn<QLIN_INT8, false>, grid, block, 0, st, 1, (const uint16_t *)x, s, q, K)
             : launch_kernel(k_quantize_act_dyn<QLIN_E4M3, false>, grid, block, 0, st, 1, (const uint16_t *)x, s, q, K);
}
}  // namespace qlin
