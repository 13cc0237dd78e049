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

// fp32 -> BF16 bit pattern, round to nearest even.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// One quantization step q = Q(x / s): IEEE binary32 division, then
// INT8: round half to even + clamp to [-127,127];  E4M3: saturating RNE cast.
template <int QT>
__device__ __forceinline__ uint8_t quantize_one(float x, float s) {
  float v = __fdiv_rn(x, s);
  if constexpr (QT == QLIN_INT8) {
    float r = fminf(fmaxf(rintf(v), -127.0f), 127.0f);
    return (uint8_t)(int8_t)__float2int_rn(r);
  } else {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
  }
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
