// Mixed KV-cache quantization kernels: keys as INT8 with one float16 scale per
// 32 head_dim elements, values as E4M3 with one float16 scale per token and kv
// head ("Nano-vLLM-MoE" README, section "KV cache compression": mixed K int8 +
// V FP8, K group 32, float16 scales, dynamic per-token quantization).
//
// Store mapping: a warp works on one token and four of its kv heads at a time
// (an "item"); lanes 8j..8j+7 hold head j of the item, lane 8j+i holds
// elements [i*E, (i+1)*E) of that head row, E = D/8 (4, 8, 16 or 32).  So a
// 32-element key group is 32/E adjacent lanes (a single lane for D = 256) and
// a value head is 8 lanes: each lane computes one key-group scale and one
// value scale per item, and the abs-max reductions are at most 3 shuffles.  A
// warp's load of an item's key (or value) rows is 4 * D * 2 contiguous bytes.
// The load kernel maps a head row onto the whole warp instead (see there).
// Pure HBM streams: no shared memory, no waits.
#include "common.cuh"
#include "kernels.h"

#include <cuda_fp16.h>

#include <algorithm>

namespace qlin {

namespace {

constexpr int kTokensPerBlock = 8;  // 8 warps of 32 threads
constexpr int kHeadsPerItem = 4;    // heads of one token a warp handles at once
constexpr int kLanesPerHead = 8;

// N 32-bit words at an address aligned to 4*min(N,4) bytes.
template <int N>
__device__ __forceinline__ void load_words(const void *p, uint32_t (&w)[N]) {
  if constexpr (N == 1) {
    w[0] = __ldg(reinterpret_cast<const uint32_t *>(p));
  } else if constexpr (N == 2) {
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
    w[0] = v.x, w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p) + i);
      w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
    }
  }
}

template <int N>
__device__ __forceinline__ void store_words(void *p, const uint32_t (&w)[N]) {
  if constexpr (N == 1) {
    *reinterpret_cast<uint32_t *>(p) = w[0];
  } else if constexpr (N == 2) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
  } else {
#pragma unroll
    for (int i = 0; i < N / 4; ++i)
      reinterpret_cast<uint4 *>(p)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
}

// Max over aligned groups of W lanes (W a power of two <= 32).
template <int W>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// float16 scale of a group: RN_fp16(fl32(amax / qmax)), saturating at 65504;
// 1.0 when the cast gives zero.
__device__ __forceinline__ uint16_t scale16(float amax, float qmax) {
  // qmax is 127 or 448: its reciprocal is a compile-time constant and the
  // quotient amax / qmax the correctly rounded one (qlin::quotient)
  const Scale q{qmax, 1.0f / qmax, true};
  const float s32 = fminf(quotient<true>(amax, q), 65504.0f);
  uint16_t h = __half_as_ushort(__float2half_rn(s32));
  return (h & 0x7FFFu) ? h : (uint16_t)0x3C00u;
}

__device__ __forceinline__ float half_bits_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// INT8 code of a quotient v: clamp to [-127,127], then add 1.5 * 2^23.  The
// sum lies in [2^23, 2^24), where the float spacing is 1, so the addition
// rounds v half to even and the low byte of the sum's bit pattern is the code
// in two's complement.
__device__ __forceinline__ uint32_t int8_code_word(float v) {
  return __float_as_uint(__fadd_rn(fminf(fmaxf(v, -127.0f), 127.0f), 0x1.8p23f));
}

// Four low bytes -> one word (byte i from the i-th argument).
__device__ __forceinline__ uint32_t pack4_low(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// Four saturating E4M3 codes, two per conversion instruction (byte i from the
// i-th argument).
__device__ __forceinline__ uint32_t e4m3_pack4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return __byte_perm(lo, hi, 0x5410);
}

// Resident CTAs per SM the register budget is sized for (as many as fit
// without spills: 4 CTAs = 32 warps allow 64 registers a thread, 3 allow 85,
// 2 allow 128).
constexpr int min_blocks(int e) { return e >= 32 ? 2 : e >= 16 ? 3 : 4; }

// ---------------------------------------------------------------------------
// Store.  Persistent: warp w of W handles tokens w, w + W, ..., each in items
// of kHeadsPerItem heads.  The next item's rows are loaded before the current
// item is quantized, so loads overlap the arithmetic.
// ---------------------------------------------------------------------------
template <int E>
struct StoreItem {
  uint32_t k[E / 2], v[E / 2];  // E BF16 of the lane's key / value row piece
  int64_t slot;
};

template <int E>
__device__ __forceinline__ void store_fetch(StoreItem<E> &it, int64_t t, int h, bool active,
                                            const uint16_t *__restrict__ k, int64_t ldk,
                                            const uint16_t *__restrict__ v, int64_t ldv,
                                            const int64_t *__restrict__ slots, int sub) {
  constexpr int D = 8 * E;
  it.slot = __ldg(slots + t);
#pragma unroll
  for (int i = 0; i < E / 2; ++i) it.k[i] = it.v[i] = 0u;
  if (active) {
    load_words<E / 2>(k + t * ldk + (int64_t)h * D + sub * E, it.k);
    load_words<E / 2>(v + t * ldv + (int64_t)h * D + sub * E, it.v);
  }
}

template <int E>
__global__ void __launch_bounds__(32 * kTokensPerBlock, min_blocks(E)) k_kv_store_mixed(
    const uint16_t *__restrict__ k, int64_t ldk, const uint16_t *__restrict__ v, int64_t ldv,
    const int64_t *__restrict__ slots, int64_t T, int H, int64_t num_slots, uint8_t *__restrict__ kc,
    uint16_t *__restrict__ ks, uint8_t *__restrict__ vc, uint16_t *__restrict__ vs, unsigned *status) {
  constexpr int D = 8 * E;
  constexpr int GL = E >= 32 ? 1 : 32 / E;  // lanes per 32-element key group
  static_assert(E <= 32, "a lane holds at most one 32-element key group");
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int j = lane / kLanesPerHead, sub = lane % kLanesPerHead;
  const int64_t nwarps = (int64_t)gridDim.x * kTokensPerBlock;
  int64_t t = (int64_t)blockIdx.x * kTokensPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  int h0 = 0;
  StoreItem<E> cur, nxt;
  store_fetch<E>(cur, t, h0 + j, h0 + j < H, k, ldk, v, ldv, slots, sub);
  while (true) {
    // the item after (t, h0): the next heads of this token, or the next token
    int64_t tn = t;
    int hn = h0 + kHeadsPerItem;
    if (hn >= H) {
      hn = 0;
      tn = t + nwarps;
    }
    if (tn < T) store_fetch<E>(nxt, tn, hn + j, hn + j < H, k, ldk, v, ldv, slots, sub);
    const int64_t slot = cur.slot;
    const int h = h0 + j;
    if (slot >= num_slots) {
      if (lane == 0 && h0 == 0) set_status(status, QLIN_ERR_INVALID_ARG);
    } else if (slot >= 0) {
      // lanes of heads past H compute on zeros and store nothing (the warp
      // stays converged for the shuffles)
      float kf[E], vf[E];
#pragma unroll
      for (int i = 0; i < E / 2; ++i) {
        kf[2 * i] = bf16_bits_to_f32(cur.k[i] & 0xFFFFu);
        kf[2 * i + 1] = __uint_as_float(cur.k[i] & 0xFFFF0000u);
        vf[2 * i] = bf16_bits_to_f32(cur.v[i] & 0xFFFFu);
        vf[2 * i + 1] = __uint_as_float(cur.v[i] & 0xFFFF0000u);
      }
      float ka = 0.0f, va = 0.0f;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        ka = fmaxf(ka, fabsf(kf[i]));
        va = fmaxf(va, fabsf(vf[i]));
      }
      ka = group_max<GL>(ka);
      va = group_max<kLanesPerHead>(va);
      const uint16_t ks16 = scale16(ka, kQmaxInt8);
      const uint16_t vs16 = scale16(va, kQmaxE4m3);
      const Scale ksc = make_scale(half_bits_to_f32(ks16)), vsc = make_scale(half_bits_to_f32(vs16));
      uint32_t kq[E / 4], vq[E / 4];
#pragma unroll
      for (int i = 0; i < E / 4; ++i) {
        kq[i] = pack4_low(int8_code_word(quotient<true>(kf[4 * i], ksc)),
                          int8_code_word(quotient<true>(kf[4 * i + 1], ksc)),
                          int8_code_word(quotient<true>(kf[4 * i + 2], ksc)),
                          int8_code_word(quotient<true>(kf[4 * i + 3], ksc)));
        vq[i] = e4m3_pack4(quotient<true>(vf[4 * i], vsc), quotient<true>(vf[4 * i + 1], vsc),
                           quotient<true>(vf[4 * i + 2], vsc), quotient<true>(vf[4 * i + 3], vsc));
      }
      if (h < H) {
        const int64_t base = slot * H + h;
        store_words<E / 4>(kc + base * D + sub * E, kq);
        store_words<E / 4>(vc + base * D + sub * E, vq);
        if (sub % GL == 0) ks[base * (D / 32) + sub / GL] = ks16;
        if (sub == 0) vs[base] = vs16;
      }
    }
    if (tn >= T) break;
    t = tn;
    h0 = hn;
    cur = nxt;
  }
}

// ---------------------------------------------------------------------------
// Load: one warp per token, kHeadsPerItem heads at a time; all code and scale
// loads of an item are issued before any is used.  Unlike the store, a head
// row spans the whole warp (lane l holds elements [l*L, (l+1)*L), L = D/32):
// the load writes twice the bytes it reads, and with this mapping every store
// instruction writes whole contiguous lines (32 * 2L bytes of one row).
// ---------------------------------------------------------------------------
template <int L>
struct LoadWords;  // L codes / L BF16 values as one vector
template <>
struct LoadWords<1> {
  using C = uint8_t;
  using B = uint16_t;
};
template <>
struct LoadWords<2> {
  using C = uint16_t;
  using B = uint32_t;
};
template <>
struct LoadWords<4> {
  using C = uint32_t;
  using B = uint2;
};
template <>
struct LoadWords<8> {
  using C = uint2;
  using B = uint4;
};

template <int L>
__device__ __forceinline__ typename LoadWords<L>::B dequant_row(typename LoadWords<L>::C kc, float s, bool e4m3) {
  union {
    typename LoadWords<L>::C v;
    uint8_t b[L];
  } in;
  union {
    typename LoadWords<L>::B v;
    uint16_t h[L];
  } out;
  in.v = kc;
#pragma unroll
  for (int i = 0; i < L; ++i) {
    const float c = e4m3 ? code_to_f32<QLIN_E4M3>(in.b[i]) : code_to_f32<QLIN_INT8>(in.b[i]);
    out.h[i] = f32_to_bf16_bits(c * s);
  }
  return out.v;
}

template <int L>
__global__ void __launch_bounds__(32 * kTokensPerBlock, L >= 8 ? 4 : 6) k_kv_load_mixed(
    const int64_t *__restrict__ slots, int64_t T, int H, int64_t num_slots, const uint8_t *__restrict__ kc,
    const uint16_t *__restrict__ ks, const uint8_t *__restrict__ vc, const uint16_t *__restrict__ vs,
    uint16_t *__restrict__ ko, uint16_t *__restrict__ vo, unsigned *status) {
  constexpr int D = 32 * L;
  constexpr int GL = 32 / L;  // lanes per 32-element key group
  constexpr int HF = kHeadsPerItem;
  using C = typename LoadWords<L>::C;
  using B = typename LoadWords<L>::B;
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kTokensPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  const int64_t slot = __ldg(slots + t);
  const bool ok = slot >= 0 && slot < num_slots;
  if (slot >= num_slots && lane == 0) set_status(status, QLIN_ERR_INVALID_ARG);
  for (int h0 = 0; h0 < H; h0 += HF) {
    C kw[HF], vw[HF];
    uint16_t ksh[HF], vsh[HF];
#pragma unroll
    for (int j = 0; j < HF; ++j) {
      kw[j] = vw[j] = C{};
      ksh[j] = vsh[j] = 0;
      if (ok && h0 + j < H) {
        const int64_t base = slot * H + h0 + j;
        kw[j] = __ldg(reinterpret_cast<const C *>(kc + base * D) + lane);
        vw[j] = __ldg(reinterpret_cast<const C *>(vc + base * D) + lane);
        ksh[j] = __ldg(ks + base * (D / 32) + lane / GL);
        vsh[j] = __ldg(vs + base);
      }
    }
    // code * scale is exact in fp32 (at most 8 x 11 significant bits), so the
    // BF16 cast is the only rounding; a missing slot gives 0 * 0 = +0.
#pragma unroll
    for (int j = 0; j < HF; ++j) {
      if (h0 + j < H) {
        const int64_t row = t * H + h0 + j;
        reinterpret_cast<B *>(ko + row * D)[lane] = dequant_row<L>(kw[j], half_bits_to_f32(ksh[j]), false);
        reinterpret_cast<B *>(vo + row * D)[lane] = dequant_row<L>(vw[j], half_bits_to_f32(vsh[j]), true);
      }
    }
  }
}

template <int E>
cudaError_t store_e(const KvArgs &a, unsigned *status, int sms, cudaStream_t st) {
  // persistent: as many CTAs as are resident at once (or fewer for small T)
  const int64_t need = (a.T + kTokensPerBlock - 1) / kTokensPerBlock;
  const dim3 grid((unsigned)std::min<int64_t>(need, (int64_t)sms * min_blocks(E)));
  return launch_kernel(k_kv_store_mixed<E>, grid, dim3(32 * kTokensPerBlock), 0, st, 1, (const uint16_t *)a.k,
                       a.ldk, (const uint16_t *)a.v, a.ldv, a.slots, a.T, (int)a.H, a.num_slots,
                       (uint8_t *)a.k_cache, (uint16_t *)a.k_scale, (uint8_t *)a.v_cache, (uint16_t *)a.v_scale,
                       status);
}

template <int L>
cudaError_t load_l(const KvArgs &a, unsigned *status, cudaStream_t st) {
  const dim3 grid((unsigned)((a.T + kTokensPerBlock - 1) / kTokensPerBlock));
  return launch_kernel(k_kv_load_mixed<L>, grid, dim3(32 * kTokensPerBlock), 0, st, 1, a.slots, a.T, (int)a.H,
                       a.num_slots, (const uint8_t *)a.k_cache, (const uint16_t *)a.k_scale,
                       (const uint8_t *)a.v_cache, (const uint16_t *)a.v_scale, (uint16_t *)a.k_out,
                       (uint16_t *)a.v_out, status);
}

}  // namespace

cudaError_t launch_kv_store(const KvArgs &a, unsigned *status, int sms, cudaStream_t st) {
  switch (a.D) {
    case 32: return store_e<4>(a, status, sms, st);
    case 64: return store_e<8>(a, status, sms, st);
    case 128: return store_e<16>(a, status, sms, st);
    case 256: return store_e<32>(a, status, sms, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_kv_load(const KvArgs &a, unsigned *status, cudaStream_t st) {
  switch (a.D) {
    case 32: return load_l<1>(a, status, st);
    case 64: return load_l<2>(a, status, st);
    case 128: return load_l<4>(a, status, st);
    case 256: return load_l<8>(a, status, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qlin
