// W8A16 linear (BF16 activations, 8-bit weight codes with per-channel scales)
// on the FP8 tensor cores, with no per-code conversion of the weights
// ("Nano-vLLM-MoE" README, "FP8 W8A16 weight-only quantization": FP8 weights
// dequantized to BF16 for a BF16 x BF16 product with fp32 accumulation).
//
// The weight stream is the cost of a small-batch linear, and turning every code
// into BF16 before a BF16 MMA costs more issue slots than the stream leaves.
// Instead the activations, which are few, are put into the weights' format.
// Each token row x_m gets a power-of-two scale s_m (the least with
// 448 s_m >= max |x_m|), and every element v = x / s_m is written as two E4M3
// terms in one of two bands:
//   band A, |v| >= 2^-6:  x1 = RN_e4m3(v),  x2 = RN_e4m3(16 (v - x1)),
//                         v = x1 + x2 / 16;
//   band B, |v| <  2^-6:  with v' = 2^14 v,
//                         x3 = RN_e4m3(v'), x4 = RN_e4m3(16 (v' - x3)),
//                         v = 2^-14 (x3 + x4 / 16);
// the terms of the other band are zero.  A band's split is exact whenever its
// value (v, or v') is at least 2^-6 in magnitude: the first term keeps the
// leading 4 significant bits, the remainder is a multiple of 2^(e-7) below
// 2^(e-3) (e the exponent of the value, e >= -6), so 16 times it has at most 4
// significant bits from 2^(e-3) >= 2^-9 upwards, which E4M3 holds (the
// subnormals reach down to 2^-9; a BF16 value has 8 significant bits).  So
// every element with |x| >= 2^-20 s_m, which includes everything within
// 2^-28.8 of the row's maximum, is represented exactly; the rest keep an
// absolute error of at most 2^-28 s_m (below 2^-35.8 of the row's maximum).
// A row whose few "massive" channels dwarf the others by 2^20 therefore still
// has its ordinary elements exact.  Then
//   sum_k w[n,k] x[m,k] = s_m (A1 + A2 / 16 + 2^-14 (A3 + A4 / 16)),
//   Aj = sum_k w[n,k] xj[m,k],
// four FP8 products read straight from the weight codes: one E4M3 MMA with the
// four terms of every token as 4 x TT columns of the B operand (swap AB: the
// weight rows are the MMA's 128 rows, so one token still fills the tensor
// core's M), and an epilogue that forms s_m s_w[n] (...) + b[n].
// INT8 weights: the same with the INT8 codes read as E4M3 would be wrong, so
// this path is E4M3 only.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace qlin {
using namespace tc;
namespace {

// ------------------------------------------------------------ activation split
// A token row is split by one cluster of at most kSplitMaxChunks CTAs, each over
// its own chunk of at most kSplitMaxPer 16-byte pieces per thread.
constexpr int kSplitThreads = 256, kSplitMaxChunks = 8, kSplitMaxPer = 8;
constexpr int kSplitTerms = 4;  // x1, x2 (band A) and x3, x4 (band B)

// Least power of two s with 448 s >= a (a > 0), from the exponent bits alone:
// a = f 2^e with f in [1, 2); 448 = 1.75 2^8, so s = 2^(e-8) when f <= 1.75,
// else 2^(e-7).  At least 2^-126, so that 1/s is finite (a row that small still
// fits: 448 2^-126 exceeds every value below 2^-117).
__device__ __forceinline__ float split_scale(float a) {
  if (!(a > 0.0f)) return 1.0f;
  int e;
  const float f = 2.0f * frexpf(a, &e);  // a = f 2^(e-1), f in [1, 2)
  return ldexpf(1.0f, max(-126, (e - 1) - (f <= 1.75f ? 8 : 7)));
}

__device__ __forceinline__ float absmax8(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float a = 0.0f;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    a = fmaxf(a, fmaxf(fabsf(bf16_bits_to_f32(w[e] & 0xFFFFu)), fabsf(bf16_bits_to_f32(w[e] >> 16))));
  return a;
}

// The two-band split of two BF16 values (one 32-bit word) scaled by r = 1/s (a
// power of two, so x * r is exact): c[q] holds the two codes of term q + 1
// (element 0 in the low byte).
__device__ __forceinline__ void split_pair(uint32_t word, float r, uint32_t (&c)[kSplitTerms]) {
  float v[2] = {bf16_bits_to_f32(word & 0xFFFFu) * r, bf16_bits_to_f32(word >> 16) * r};
  // band B: the element scaled by 2^14 (exact), split the same way into x3, x4
  bool lo[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    lo[h] = fabsf(v[h]) < 0.015625f;  // |v| < 2^-6
    if (lo[h]) v[h] *= 16384.0f;
  }
  const __nv_fp8x2_storage_t h1 = __nv_cvt_float2_to_fp8x2(make_float2(v[0], v[1]), __NV_SATFINITE, __NV_E4M3);
  const float2 f1 = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h1, __NV_E4M3)));
  // the remainders are exact in fp32; times 16 they fit E4M3 (see the file's head)
  const __nv_fp8x2_storage_t h2 =
      __nv_cvt_float2_to_fp8x2(make_float2(16.0f * (v[0] - f1.x), 16.0f * (v[1] - f1.y)), __NV_SATFINITE, __NV_E4M3);
  // each element's two codes go to its band's pair of terms, zero to the other pair
  const uint32_t a = (lo[0] ? 0x0000u : 0x00FFu) | (lo[1] ? 0x0000u : 0xFF00u), b = ~a & 0xFFFFu;
  c[0] = (uint32_t)h1 & a, c[1] = (uint32_t)h2 & a, c[2] = (uint32_t)h1 & b, c[3] = (uint32_t)h2 & b;
}

// Token row m: one cluster of gridDim.x CTAs (or one CTA without a cluster),
// CTA c over pieces [c P, c P + P) of the row (P = `per` 16-byte pieces of 8
// elements; each thread holds up to kSplitMaxPer of them in registers).  Each CTA takes the abs-max of its own
// chunk and stores it into every CTA of the cluster (distributed shared
// memory); after one cluster barrier each CTA has the row's maximum, so the
// row is read once in all.  Each CTA then writes its chunk's four E4M3 terms
// into the B-operand layout: token tile j (tt tokens) owns rows
// [4 tt j, 4 tt j + 4 tt) of xs, the x1 rows of its tokens first, then x2, x3
// and x4.
__global__ void __launch_bounds__(kSplitThreads) k_w8a16_split(const uint16_t *__restrict__ x, int M, int K,
                                                               int tt, int per, uint8_t *__restrict__ xs,
                                                               float *__restrict__ xscale, unsigned *status) {
  __shared__ float wmax[kSplitThreads / 32];
  __shared__ float cmax[kSplitMaxChunks];  // every chunk's maximum, stored by its CTA
  // the chunks exchange their maxima through the cluster's shared memory: without
  // that cluster shape, report and leave before anything is read or written
  const int C = gridDim.x, c = blockIdx.x;
  if ((int)cluster_nctarank() != C) {
    if (threadIdx.x == 0 && c == 0) set_status(status, QLIN_ERR_UNSUPPORTED);
    return;
  }
  const int m = blockIdx.y, n8 = K / 8;  // K % 16 == 0
  const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)m * K);
  const int u0 = c * per, u1 = min(n8, u0 + per);
  // While the previous kernel finishes: pull this chunk of the row into L2 (a
  // prefetch returns nothing, so it reads no value before the wait below), so
  // that the loads after the wait do not queue behind the next linear's
  // weight traffic in HBM.
#pragma unroll
  for (int i = 0; i < kSplitMaxPer; ++i) {
    const int u = u0 + (int)threadIdx.x + i * kSplitThreads;
    if (u < u1 && (u & 7) == 0) prefetch_l2(row + u);  // one per 128-byte line
  }
  // The FP8 linear that follows may start at once: before its own wait for this
  // kernel it only arms barriers and loads weight tiles, so its CTAs take the
  // SMs that the previous linear frees during its tail.  Nothing here is
  // read or written before the previous kernel has completed.
  pdl_trigger();
  pdl_wait();
  uint4 v[kSplitMaxPer];
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < kSplitMaxPer; ++i) {  // all of this thread's loads in flight at once
    const int u = u0 + (int)threadIdx.x + i * kSplitThreads;
    v[i] = u < u1 ? __ldg(row + u) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < kSplitMaxPer; ++i) a = fmaxf(a, absmax8(v[i]));
  a = warp_max(a);
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = a;
  __syncthreads();
  if (C == 1) {  // the whole row in this CTA: no exchange
    a = wmax[0];
#pragma unroll
    for (int w = 1; w < kSplitThreads / 32; ++w) a = fmaxf(a, wmax[w]);
  } else {
    if (threadIdx.x < C) {  // this chunk's maximum into CTA threadIdx.x of the cluster
      float cm = wmax[0];
#pragma unroll
      for (int w = 1; w < kSplitThreads / 32; ++w) cm = fmaxf(cm, wmax[w]);
      st_dsmem_f32(map_peer_smem(smem_u32(&cmax[c]), threadIdx.x), cm);
    }
    cluster_sync();  // every chunk's maximum has arrived
    a = cmax[0];
    for (int q = 1; q < C; ++q) a = fmaxf(a, cmax[q]);
  }
  const float s = split_scale(a), r = 1.0f / s;  // powers of two: exact
  if (c == 0 && threadIdx.x == 0) xscale[m] = s;
  const int j = m / tt, t = m % tt;
  uint8_t *x1 = xs + ((size_t)kSplitTerms * tt * j + t) * K;
  const size_t term = (size_t)tt * K;  // x2, x3, x4 follow, tt rows apart
#pragma unroll
  for (int i = 0; i < kSplitMaxPer; ++i) {
    const int u = u0 + (int)threadIdx.x + i * kSplitThreads;
    if (u >= u1) break;
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t cw[4][kSplitTerms];  // codes of the four words' terms, two per 16 bits
#pragma unroll
    for (int e = 0; e < 4; ++e) split_pair(w[e], r, cw[e]);
#pragma unroll
    for (int q = 0; q < kSplitTerms; ++q)
      *reinterpret_cast<uint2 *>(x1 + q * term + 8 * (size_t)u) =
          make_uint2(cw[0][q] | (cw[1][q] << 16), cw[2][q] | (cw[3][q] << 16));
  }
}

// ------------------------------------------------------------ the FP8 linear
// One CTA per (weight tile, token tile, K split).  Warps: 0 = TMA producer,
// 1 = TMEM allocator and MMA issuer, 2..5 = epilogue (TMEM lane quadrants
// 2, 3, 0, 1).  A weight tile is 128 rows (plain) or 64 gate rows and their 64
// up rows (merged gate_up).  The K splits of a tile form a cluster: each CTA
// leaves its fp32 partial tile in shared memory (the drained ring) and the
// cluster sums them in rank order through distributed shared memory, each CTA
// finishing a slice of the outputs.
// The B operand (the four E4M3 terms of every token of the tile) comes from
// k_w8a16_split through the workspace, with one power-of-two scale per token
// row; the epilogue folds that scale into the partial tile, so the cluster's
// sum of the partials needs no per-token factor.
// The token tile tt (4, 8 or 16 up to TMAX = 16; 32 for TMAX = 32) is chosen
// at run time: the fewer the tokens, the smaller each stage's B tile, so the
// deeper the ring and the more weight tiles stream in before the wait for the
// split.
template <int TMAX>
struct W8F8Cfg {
  static constexpr int BM = 128, BK = 128, NB_MAX = kSplitTerms * TMAX;
  static constexpr int A_BYTES = BM * BK;
  static __host__ __device__ constexpr int stage_bytes(int tt) { return A_BYTES + kSplitTerms * tt * BK; }
  // The ring depth is a launch parameter; the barriers follow the ring, then
  // the tile's per-row weight scales and biases and the per-token scales.
  static constexpr int MAX_STAGES = 14, BAR_BYTES = 256, AUX_BYTES = (2 * BM + 32) * 4;
  static constexpr int THREADS = 192;
  static constexpr uint32_t TMEM_COLS = NB_MAX;  // 64 or 128, a power of two
  static constexpr int smem_bytes(int tt, int stages) {
    return stages * stage_bytes(tt) + BAR_BYTES + AUX_BYTES + 1024;
  }
  static_assert(TMAX == 16 || TMAX == 32, "token tile bound");
  static_assert((2 * MAX_STAGES + 1) * 8 + 8 <= BAR_BYTES, "barriers");
  static_assert(stage_bytes(4) % 1024 == 0, "stage alignment (128-byte swizzle atoms)");
};

struct W8F8Params {
  int M, N, K;  // N: output channels (I for the merged gate_up)
  int glu;
  int ntiles, splits, stages;
  int tt;  // tokens per tile
  const float *w_scale;
  const float *x_scale;  // per token, from the split
  const uint16_t *bias;
  uint16_t *y;
  unsigned *status;
};

__device__ __forceinline__ uint8_t *align1k(uint8_t *p) {
  return (uint8_t *)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

template <int TMAX>
__global__ void __launch_bounds__(W8F8Cfg<TMAX>::THREADS, 1)
    k_w8a16_f8(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x, W8F8Params p) {
  using C = W8F8Cfg<TMAX>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1k(smem_raw);
  const int NS = p.stages, tt = p.tt, NB = kSplitTerms * tt, STAGE = C::stage_bytes(tt);
  uint64_t *full = (uint64_t *)(smem + NS * STAGE), *empty = full + NS, *acc_full = empty + NS;
  uint32_t *tmem_slot = (uint32_t *)(acc_full + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
  float *rsc = (float *)(smem + NS * STAGE + C::BAR_BYTES), *rbi = rsc + C::BM, *xsc = rbi + C::BM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.splits;
  // the K splits of a tile reduce through their cluster's shared memory: without
  // that cluster shape, report and leave before any barrier, TMEM or peer is touched
  if (S > 1 && (int)cluster_nctarank() != S) {
    if (threadIdx.x == 0) set_status(p.status, QLIN_ERR_UNSUPPORTED);
    return;
  }
  const int split = blockIdx.z, tile = blockIdx.x % p.ntiles, tj = blockIdx.x / p.ntiles;
  const int KB = (p.K + C::BK - 1) / C::BK, kb0 = split * KB / S, kb1 = (split + 1) * KB / S, nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  if (warp == 0) {  // ------------------------------- TMA producer
    if (lane == 0) {
      auto load_w = [&](int i) {
        uint8_t *st = smem + (i % NS) * STAGE;
        const int k = (kb0 + i) * C::BK;
        if (p.glu) {  // 64 gate rows, then their 64 up rows
          tma_load_2d(&tm_w, &full[i % NS], st, k, tile * 64);
          tma_load_2d(&tm_w, &full[i % NS], st + 64 * C::BK, k, p.N + tile * 64);
        } else {
          tma_load_2d(&tm_w, &full[i % NS], st, k, tile * C::BM);
        }
      };
      auto load_x = [&](int i) {
        tma_load_2d(&tm_x, &full[i % NS], smem + (i % NS) * STAGE + C::A_BYTES, (kb0 + i) * C::BK, tj * NB);
      };
      // The weight tiles of the first stages are loaded before the wait for the
      // previous kernel: weights are never written by a kernel that lets this
      // one start early (the weight quantizer lets no later kernel start before
      // it completes).  The activation terms follow the wait.
      const int pre = nkb < NS ? nkb : NS;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], STAGE);
        load_w(i);
      }
      pdl_wait();
      int i = 0;
      for (; i < nkb; ++i) {
        const int s = i % NS;
        if (i >= NS && !mbar_wait(&empty[s], ((i / NS) & 1) ^ 1, abort_flag)) {
          *abort_flag = 1;
          break;
        }
        if (i >= pre) {  // stages past the ones armed before the wait
          mbar_arrive_expect_tx(&full[s], STAGE);
          load_w(i);
        }
        load_x(i);
      }
      if (*abort_flag) drain_ring(full, NS, i > pre ? i : pre, NS);  // armed stages land before the CTA leaves
    }
  } else if (warp == 1) {  // ------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = umma_idesc(0, 0, C::BM, NB);
      bool ok = true;
      int i = 0;
      for (; i < nkb; ++i) {
        const int s = i % NS;
        if (!mbar_wait(&full[s], (i / NS) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + s * STAGE);
        const uint64_t ad = umma_desc_sw128(a), bd = umma_desc_sw128(a + C::A_BYTES);
#pragma unroll
        for (int j = 0; j < 4; ++j)  // K = 32 codes per instruction
          mma_fp8(tmem, ad + 2 * j, bd + 2 * j, idesc, (i > 0 || j > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
      }
      if (ok) mma_commit(acc_full);
      // no commit arrival may land after the CTA has left (bounded, also on abort)
      if (i > 0) ok = mbar_wait_drain(&empty[(i - 1) % NS], ((i - 1) / NS) & 1) && ok;
      if (!ok) *abort_flag = 1;
    }
  } else {  // ------------------------------------- epilogue: accumulators -> partial tile
    const int q4 = warp & 3, r = q4 * 32 + lane;  // TMEM lane = weight row of the tile
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    // While the main loop runs: this row's weight scale and bias (weights, so
    // readable before the wait), then, after it, the tile's token scales.
    {
      const int ch = p.glu ? (r < 64 ? tile * 64 + r : p.N + tile * 64 + (r - 64)) : tile * C::BM + r;
      const bool live = p.glu || ch < p.N;
      rsc[r] = live ? __ldg(p.w_scale + ch) : 0.0f;
      rbi[r] = live && p.bias ? bf16_bits_to_f32(__ldg(p.bias + ch)) : 0.0f;
    }
    bool ok = true;
    pdl_wait();  // the split's scales are complete from here on
    const int m0 = tj * tt, e = threadIdx.x - 64;
    if (e < tt) xsc[e] = m0 + e < p.M ? __ldg(p.x_scale + m0 + e) : 0.0f;
    bar_sync_named(1, 128);  // the four epilogue warps
    ok = ok && mbar_wait(acc_full, 0, abort_flag);
    tc_fence_after();
    if (__all_sync(0xffffffffu, ok && !*abort_flag)) {  // tcgen05.ld is warp-collective
      float *part = reinterpret_cast<float *>(smem);   // the ring is drained: every MMA has read it
#pragma unroll 1
      for (int c = 0; c < tt; c += 16) {
        uint32_t a1[16], a2[16], a3[16], a4[16];  // x1..x4 products of tokens c..c+15 (c..tt-1 used)
        tmem_ld16(tmem + lane_base + c, a1);
        tmem_ld16(tmem + lane_base + tt + c, a2);
        tmem_ld16(tmem + lane_base + 2 * tt + c, a3);
        tmem_ld16(tmem + lane_base + 3 * tt + c, a4);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          if (c + t >= tt) break;
          const float band_a = fmaf(__uint_as_float(a2[t]), 0.0625f, __uint_as_float(a1[t]));
          const float band_b = fmaf(__uint_as_float(a4[t]), 0.0625f, __uint_as_float(a3[t]));
          part[(c + t) * C::BM + r] = xsc[c + t] * fmaf(band_b, 6.103515625e-05f, band_a);  // 2^-14
        }
      }
    } else {
      ok = false;
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (S > 1) cluster_sync();  // every partial tile of the cluster is written

  // ------------------------------------------- sum over the splits, finish the outputs
  // this CTA finishes items [e0, e1) of the tile: an item is 4 consecutive rows
  // (channels) of one token, read as one 16-byte piece from each CTA of the
  // cluster in rank order (deterministic); consecutive threads take consecutive
  // items of one token, so the stores are coalesced
  pdl_wait();  // y belongs to the previous kernels from here on
  {
    const int rows = p.glu ? 64 : C::BM, R4 = rows / 4, E = tt * R4;
    const int e0 = split * E / S, e1 = (split + 1) * E / S;
    const uint32_t pbase = smem_u32(smem);
    auto sum4 = [&](int t, int row) {
      if (S == 1) return *reinterpret_cast<const float4 *>(smem + 4 * (t * C::BM + row));
      const uint32_t a = pbase + 4u * (uint32_t)(t * C::BM + row);
      uint4 u[8];  // every peer's piece in flight at once, then the sum in rank order
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < S) u[q] = ld_dsmem_v4(map_peer_smem(a, (uint32_t)q));
      float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < S)
          v.x += __uint_as_float(u[q].x), v.y += __uint_as_float(u[q].y), v.z += __uint_as_float(u[q].z),
              v.w += __uint_as_float(u[q].w);
      return v;
    };
    for (int e = e0 + (int)threadIdx.x; e < e1; e += C::THREADS) {
      const int t = e / R4, rr = (e - t * R4) * 4, m = tj * tt + t;
      if (m >= p.M) continue;
      float o[4];
      int n;
      if (p.glu) {
        n = tile * 64 + rr;
        const float4 g4 = sum4(t, rr), u4 = sum4(t, 64 + rr);
        const float gs[4] = {g4.x, g4.y, g4.z, g4.w}, us[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float g = fmaf(gs[i], rsc[rr + i], rbi[rr + i]);
          const float u = fmaf(us[i], rsc[64 + rr + i], rbi[64 + rr + i]);
          o[i] = silu_f(g) * u;
        }
      } else {
        n = tile * C::BM + rr;
        if (n >= p.N) continue;  // N % 16 == 0: the four channels are all in or all out
        const float4 v4 = sum4(t, rr);
        const float vs[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = fmaf(vs[i], rsc[rr + i], rbi[rr + i]);
      }
      *reinterpret_cast<uint2 *>(p.y + (size_t)m * p.N + n) =
          make_uint2(f32_to_bf16_bits(o[0]) | ((uint32_t)f32_to_bf16_bits(o[1]) << 16),
                     f32_to_bf16_bits(o[2]) | ((uint32_t)f32_to_bf16_bits(o[3]) << 16));
    }
  }
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, QLIN_ERR_TIMEOUT);
  __syncthreads();
  if (S > 1) cluster_sync();  // no CTA leaves while a peer may still read its shared memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
            cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)q;
  });
  return fn;
}

// Row-major [rows, cols] bytes, box = 128 columns x box_rows, 128-byte swizzle.
bool map_u8(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared memory of one CTA when two share an SM (228 KB, 1 KB of it reserved per CTA).
constexpr int kCtaSmem = 113 * 1024;

template <int TMAX>
cudaError_t launch_tt(const GemmArgs &g, int tt, uint8_t *xs, float *xscale, const DeviceInfo &dev,
                      cudaStream_t st) {
  using C = W8F8Cfg<TMAX>;
  const int ttiles = (int)((g.M + tt - 1) / tt), NB = kSplitTerms * tt;
  CUtensorMap tw, tx;
  if (!map_u8(&tw, g.qw, g.glu ? 2 * g.N : g.N, g.K, g.glu ? 64 : 128) ||
      !map_u8(&tx, xs, (int64_t)ttiles * NB, g.K, NB))
    return cudaErrorInvalidValue;
  // one cluster per token row: C CTAs of about two (at most kSplitMaxPer) 16-byte
  // pieces per thread (one piece a thread, or four, measured slower)
  const int n8 = (int)(g.K / 8);
  int chunks = (n8 + 2 * kSplitThreads - 1) / (2 * kSplitThreads);
  if (chunks > kSplitMaxChunks) chunks = kSplitMaxChunks;
  const int per = (n8 + chunks - 1) / chunks;
  if (per > kSplitMaxPer * kSplitThreads) return cudaErrorInvalidValue;  // K beyond 2^17 (refused on the host)
  // a row that fits one CTA needs no cluster
  cudaError_t e =
      chunks == 1 ? launch_kernel(k_w8a16_split, dim3(1u, (unsigned)g.M), dim3(kSplitThreads), 0, st, 1u,
                                  (const uint16_t *)g.a, (int)g.M, (int)g.K, tt, per, xs, xscale, dev.status)
                  : launch_kernel_x(k_w8a16_split, dim3((unsigned)chunks, (unsigned)g.M), dim3(kSplitThreads), 0, st,
                                    (unsigned)chunks, (const uint16_t *)g.a, (int)g.M, (int)g.K, tt, per, xs, xscale,
                                    dev.status);
  if (e != cudaSuccess) return e;
  W8F8Params p;
  p.M = (int)g.M;
  p.N = (int)g.N;
  p.K = (int)g.K;
  p.glu = g.glu;
  p.tt = tt;
  p.ntiles = g.glu ? (int)(g.N / 64) : (int)((g.N + C::BM - 1) / C::BM);
  const int units = p.ntiles * ttiles, KB = (int)((g.K + C::BK - 1) / C::BK);
  p.splits = w8a16_f8_splits(units, KB, dev.sms);
  // two CTAs to an SM: as many stages as fit beside the barriers and scales
  int stages = (kCtaSmem - C::smem_bytes(tt, 0)) / C::stage_bytes(tt);
  if (stages > C::MAX_STAGES) stages = C::MAX_STAGES;
  if (stages < 3) return cudaErrorInvalidValue;
  p.stages = stages;
  p.w_scale = g.w_scale;
  p.x_scale = xscale;
  p.bias = g.bias;
  p.y = (uint16_t *)g.y;
  p.status = dev.status;
  static const cudaError_t attr =
      cudaFuncSetAttribute(k_w8a16_f8<TMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, kCtaSmem);
  if (attr != cudaSuccess) return attr;
  return launch_kernel(k_w8a16_f8<TMAX>, dim3((unsigned)units, 1, (unsigned)p.splits), dim3(C::THREADS),
                       C::smem_bytes(tt, p.stages), st, (unsigned)p.splits, tw, tx, p);
}

}  // namespace

// Token tile.  Up to kW8A16F8MaxM = 32 tokens: beyond that the E4M3 terms of
// the tile (4 tt x 128 bytes a k-block) outweigh the weight tile they meet,
// and the BF16 path with converted weights is faster.  Up to 16 tokens the
// tile is the least of 4, 8 and 16 that holds them (k_w8a16_f8<16>).
int w8a16_f8_tt(int64_t M) { return M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : 32; }

// K splits (a cluster of at most 8 CTAs): as many as fit two CTAs to an SM,
// and at least 4 k-blocks of 128 per CTA.  A CTA's stream rate is bounded by
// its own rate of issue more than by its ring depth (measured: 5 and 11 stages
// stream alike), so more CTAs beat deeper rings.
int w8a16_f8_splits(int units, int kblocks, int sms) {
  int s = 1;
  while (s < 8 && units * (s + 1) <= 2 * sms && kblocks / (s + 1) >= 4) ++s;
  return s;
}

size_t w8a16_f8_workspace(int64_t M, int64_t K) {
  const int64_t tt = w8a16_f8_tt(M), ttiles = (M + tt - 1) / tt;
  return (size_t)((ttiles * kSplitTerms * tt * K + 255) / 256 * 256) + (size_t)((M * 4 + 255) / 256 * 256);
}

cudaError_t launch_w8a16_f8(const GemmArgs &g, void *ws, const DeviceInfo &dev, cudaStream_t st) {
  if (g.M == 0) return cudaSuccess;
  if (g.qtype != QLIN_E4M3 || g.M > kW8A16F8MaxM) return cudaErrorInvalidValue;
  const int64_t tt = w8a16_f8_tt(g.M), ttiles = (g.M + tt - 1) / tt;
  uint8_t *xs = (uint8_t *)ws;
  float *xscale = (float *)((uint8_t *)ws + (ttiles * kSplitTerms * tt * g.K + 255) / 256 * 256);
  return tt <= 16 ? launch_tt<16>(g, (int)tt, xs, xscale, dev, st) : launch_tt<32>(g, (int)tt, xs, xscale, dev, st);
}

}  // namespace qlin
