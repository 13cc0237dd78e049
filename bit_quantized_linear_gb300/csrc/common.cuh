// Shared device helpers for libqlin kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qlin.h"

namespace qlin {

constexpr float kQmaxInt8 = 127.0f;
constexpr float kQmaxE4m3 = 448.0f;

__host__ __device__ constexpr float qmax_of(int qtype) {
  return qtype == QLIN_INT8 ? kQmaxInt8 : kQmaxE4m3;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// BF16 bit pattern -> fp32 (exact).
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// Two integer-valued floats of magnitude below 2^8 (8-bit codes) as BF16,
// packed (lo in the low half).  The binary32 pattern of such a value has zeros
// in its 16 low bits, so its upper half is the exact BF16 value: one byte
// permute instead of two conversions.
__device__ __forceinline__ uint32_t pack_code_bf16x2(float lo, float hi) {
  return __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);
}

// fp32 -> BF16 bit pattern, round to nearest even.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// A quantization scale s > 0 with its correctly rounded reciprocal r = RN(1/s).
// `fast` holds when s lies in [2^-96, 2^96]: then 1/s and every intermediate of
// quotient() below stay in the normal range.
struct Scale {
  float s, r;
  bool fast;
};
__device__ __forceinline__ Scale make_scale(float s) {
  return Scale{s, __frcp_rn(s), s >= 0x1p-96f && s <= 0x1p96f};
}

// x / s correctly rounded to binary32, computed from r instead of a division
// per element, by Markstein's theorem (P. W. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): if r is within half an ulp of 1/s and q within one ulp
// of x/s, the residual x - q*s is exact in one FMA and RN(q + residual * r)
// is RN(x/s), barring overflow and underflow.  q = RN(x*r) is within one ulp.
//   - BOUNDED callers derive s from the abs-max of the very values they divide,
//     so |x/s| is about QMAX and nothing overflows.  Otherwise (a static scale
//     at run time) q is first clamped to +-2^32: every code beyond that clamps
//     or saturates anyway, and the clamp keeps the residual finite.
//   - A quotient in the subnormal range gives code 0 whatever its last bits;
//     its sign (that of x, s > 0) is restored by copysign, which also keeps
//     the sign of a zero x that the correction step would lose.
//   - Scales outside [2^-96, 2^96] take the IEEE division.
template <bool BOUNDED>
__device__ __forceinline__ float quotient(float x, const Scale &c) {
  if (!c.fast) return __fdiv_rn(x, c.s);
  float q = __fmul_rn(x, c.r);
  if constexpr (!BOUNDED) q = fminf(fmaxf(q, -0x1p32f), 0x1p32f);
  const float rem = __fmaf_rn(-q, c.s, x);
  return copysignf(__fmaf_rn(rem, c.r, q), x);
}

// One quantization step q = Q(x / s): the correctly rounded binary32 quotient,
// then INT8: round half to even + clamp to [-127,127];  E4M3: saturating RNE cast.
template <int QT, bool BOUNDED>
__device__ __forceinline__ uint8_t quantize_one(float x, const Scale &c) {
  const float v = quotient<BOUNDED>(x, c);
  if constexpr (QT == QLIN_INT8) {
    float r = fminf(fmaxf(rintf(v), -127.0f), 127.0f);
    return (uint8_t)(int8_t)__float2int_rn(r);
  } else {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
  }
}

// The INT8 code of x under a run-time (static) scale, as the integer-valued
// float the BF16 MMA consumes: the same code as quantize_one<QLIN_INT8, false>
// (the same quotient, round half to even, clamp to [-127, 127]) without the
// round trip through an integer.  The copysign of quotient() only matters for
// quotients that round to zero, and a zero code is returned as +0 either way.
__device__ __forceinline__ float quantize_i8_value(float x, const Scale &c) {
  float v;
  if (c.fast) {
    const float q = fminf(fmaxf(__fmul_rn(x, c.r), -0x1p32f), 0x1p32f);
    v = __fmaf_rn(__fmaf_rn(-q, c.s, x), c.r, q);
  } else {
    v = __fdiv_rn(x, c.s);
  }
  return fminf(fmaxf(rintf(v), -127.0f), 127.0f) + 0.0f;
}

// ------------------------------------------------ static E4M3, eight at a time
// The static E4M3 quantizer of a whole tensor (one run-time scale s) gives the
// same codes as quantize_one<QLIN_E4M3, false> for every finite input, with
// about half the instructions, which matters where the conversion shares an SM
// with a GEMM:
//   - |x| is first clamped to B, the smallest BF16 >= 512 s, two lanes at a time
//     on the packed BF16 input (min of absolute values, sign kept).  Every
//     |x| >= B has |x/s| >= 512 > 448 and saturates to +-448 either way, and
//     after the clamp x * r cannot overflow, so the quotient needs no clamp.
//   - The quotient's multiply and two FMAs run as packed f32x2 operations
//     (the same IEEE round-to-nearest operations, lane by lane).
//   - The sign of x is ORed into each code byte: for x != 0 the code already
//     carries it, and for x = -0 the correction step returns +0 and the OR
//     restores -0's code 0x80 (what the copysign of quotient() does).
// Off the fast scale range it is quantize_one itself, element by element.
struct StaticE4m3 {
  Scale c;
  uint32_t bound2;   // B in both BF16 halves
  uint64_t r2, ns2;  // (r, r) and (-s, -s) as f32x2
};
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ StaticE4m3 make_static_e4m3(float s) {
  StaticE4m3 q;
  q.c = make_scale(s);
  uint32_t b = 0x7F80u;  // +inf
  if (q.c.fast) {
    const uint32_t bits = __float_as_uint(512.0f * s);  // exact (s <= 2^96)
    b = (bits >> 16) + ((bits & 0xFFFFu) ? 1u : 0u);    // round up to BF16
  }
  q.bound2 = b | (b << 16);
  q.r2 = f32x2_pack(q.c.r, q.c.r);
  q.ns2 = f32x2_pack(-s, -s);
  return q;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// Two BF16 (one word) -> two E4M3 codes in the low 16 bits (lane 0 in byte 0);
// fast scale range only, sign of a zero not yet restored.
__device__ __forceinline__ uint32_t e4m3_static2_fast(uint32_t w, const StaticE4m3 &q) {
  uint32_t wc;
  asm("min.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(wc) : "r"(w), "r"(q.bound2));
  const uint64_t x = f32x2_pack(__uint_as_float(wc << 16), __uint_as_float(wc & 0xFFFF0000u));
  const uint64_t q0 = f32x2_mul(x, q.r2);
  const uint64_t rem = f32x2_fma(q0, q.ns2, x);
  const uint64_t q1 = f32x2_fma(rem, q.r2, q0);
  return (uint32_t)__nv_cvt_float2_to_fp8x2(
      make_float2(__uint_as_float((uint32_t)q1), __uint_as_float((uint32_t)(q1 >> 32))), __NV_SATFINITE,
      __NV_E4M3);
}
// Four BF16 (two words) -> four codes, element i in byte i.  The _fast form
// (no branch, so a caller's unrolled loop schedules freely) needs q.c.fast.
__device__ __forceinline__ uint32_t e4m3_static4_fast(uint32_t w0, uint32_t w1, const StaticE4m3 &q) {
  const uint32_t c = __byte_perm(e4m3_static2_fast(w0, q), e4m3_static2_fast(w1, q), 0x5410);
  return c | (__byte_perm(w0, w1, 0x7531) & 0x80808080u);  // the BF16 sign bits
}
__device__ __forceinline__ uint32_t e4m3_static4_exact_div(uint32_t w0, uint32_t w1, const Scale &c) {
  return (uint32_t)quantize_one<QLIN_E4M3, false>(bf16_bits_to_f32(w0 & 0xFFFFu), c) |
         ((uint32_t)quantize_one<QLIN_E4M3, false>(bf16_bits_to_f32(w0 >> 16), c) << 8) |
         ((uint32_t)quantize_one<QLIN_E4M3, false>(bf16_bits_to_f32(w1 & 0xFFFFu), c) << 16) |
         ((uint32_t)quantize_one<QLIN_E4M3, false>(bf16_bits_to_f32(w1 >> 16), c) << 24);
}

// Exact value of an 8-bit code as fp32 (every INT8 / E4M3 value is exact in fp32).
template <int QT>
__device__ __forceinline__ float code_to_f32(uint8_t c) {
  if constexpr (QT == QLIN_INT8) {
    return (float)(int8_t)c;
  } else {
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
    return __half2float(__half(h));
  }
}

// SiLU of the merged gate_up epilogue: g * sigmoid(g) = g / (1 + exp(-g)), with
// CUDA's fast exponential and division intrinsics (relative error ~2^-21, far
// below the BF16 rounding of the output).  Extremes: for g > ~88, exp(-g) is 0
// and the result is g; for g < ~-87, 1 + exp(-g) exceeds 2^126 and __fdividef
// returns 0, where the exact value is below 2^-100 in magnitude.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while the previous kernel in the
// stream is still running; pdl_wait() blocks until that kernel has completed
// and its memory is visible (a no-op without the attribute).  pdl_trigger()
// lets the next kernel start its own prologue early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Sets the device status word (first error wins).
__device__ __forceinline__ void set_status(unsigned *status, unsigned code) {
  if (status) atomicCAS(status, 0u, code);
}

}  // namespace qlin
