// Tensor-core (tcgen05) GEMMs for the quantized linear on sm_103a.
//
// k_fp8_gemm   W8A8 with E4M3 activations and weights: TMA loads both 8-bit
//              operand tiles (128-byte swizzle) into a 4-stage shared-memory
//              ring, one thread issues tcgen05.mma kind::f8f6f4 into a TMEM
//              accumulator (fp32), four epilogue warps read TMEM and apply
//              y = acc * (s_x * s_w[n]) + bias[n] -> BF16.
//              Tile: 128 tokens x BN output channels x 128 k per stage.
//
// k_w8_swap    W8A16 (INT8 or E4M3 weight codes, BF16 activations) with the
//              weights as the 128-row MMA operand ("swap AB": output channels
//              on the TMEM lanes, tokens on the MMA N dimension, 16..256), so
//              decode batches of a few tokens still fill the tensor core's M.
//              TMA streams raw 8-bit weight tiles and BF16 activation tiles;
//              four converter warps turn each raw tile into an exact BF16 tile
//              in the UMMA 128-byte-swizzle layout; one thread issues
//              tcgen05.mma kind::f16.  When there are too few output tiles to
//              fill the GPU, the K range is split over the CTAs of a cluster
//              and the fp32 partial tiles are summed in a fixed order through
//              distributed shared memory -- one kernel, deterministic, no
//              global workspace and no spinning on global flags.
//
// Warp roles (256 threads): warp 0 = TMA producer, warp 1 = TMEM allocator and
// MMA issuer, warps 4..7 = converters (k_w8_swap) and epilogue (TMEM lane
// quarter = warp % 4).  Every mbarrier wait is bounded (tc::mbar_wait); a wait
// that runs out sets the device status word and the CTA leaves through the
// same exit path (TMEM freed, cluster barriers met).
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace qlin {

using namespace tc;

// ============================================================ host: TMA maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

// Row-major [rows, cols] matrix of `esize`-byte elements; box = box_cols x box_rows.
static bool make_map(CUtensorMap *tm, const void *base, CUtensorMapDataType dt, int esize, int64_t rows,
                     int64_t cols, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * esize)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return (uint8_t *)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// ============================================================ FP8 W8A8 GEMM
struct Fp8Params {
  int M, N, K;
  const float *w_scale;
  const float *x_scale;
  const uint16_t *bias;
  uint16_t *y;
  unsigned *status;
};

template <int BN>
struct Fp8Cfg {
  static constexpr int BM = 128, BK = 128, STAGES = 4;
  static constexpr int A_BYTES = BM * BK, B_BYTES = BN * BK, STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr uint32_t IDESC = umma_idesc(0, 0, BM, BN);
};

template <int BN>
__global__ void __launch_bounds__(256, 1)
    k_fp8_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, Fp8Params p) {
  using C = Fp8Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *full = (uint64_t *)(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t *empty = full + C::STAGES;
  uint64_t *acc_full = empty + C::STAGES;
  uint32_t *tmem_slot = (uint32_t *)(acc_full + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * C::BM, n0 = blockIdx.x * BN;
  const int nkb = (p.K + C::BK - 1) / C::BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) tmem_alloc(tmem_slot, BN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {  // ---------------- TMA producer
    for (int i = 0; i < nkb; ++i) {
      const int s = i % C::STAGES;
      if (i >= C::STAGES && !mbar_wait(&empty[s], ((i / C::STAGES) & 1) ^ 1, abort_flag)) {
        *abort_flag = 1;
        break;
      }
      uint8_t *a = smem + s * C::STAGE_BYTES;
      mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
      tma_load_2d(&tm_a, &full[s], a, i * C::BK, m0);
      tma_load_2d(&tm_b, &full[s], a + C::A_BYTES, i * C::BK, n0);
    }
  } else if (warp == 1 && lane == 0) {  // ---------- MMA issuer
    bool ok = true;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % C::STAGES;
      if (!mbar_wait(&full[s], (i / C::STAGES) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a = smem_u32(smem + s * C::STAGE_BYTES);
      const uint64_t ad = umma_desc_sw128(a), bd = umma_desc_sw128(a + C::A_BYTES);
#pragma unroll
      for (int kk = 0; kk < C::BK / 32; ++kk)  // K = 32 per instruction (32 bytes)
        mma_fp8(tmem, ad + 2 * kk, bd + 2 * kk, C::IDESC, (i | kk) != 0);
      mma_commit(&empty[s]);
    }
    if (!ok) *abort_flag = 1;
    mma_commit(acc_full);
  } else if (warp >= 4) {  // ------------------------ epilogue
    const int q = warp & 3;
    const int m = m0 + q * 32 + lane;
    const bool ok = mbar_wait(acc_full, 0, abort_flag);
    tc_fence_after();
    // tcgen05.ld is warp-collective: every lane of the warp takes the same path
    if (__all_sync(0xffffffffu, ok && !*abort_flag)) {
      const float sx = __ldg(p.x_scale);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, r);
        tmem_ld_wait();
        const int nb = n0 + c * 32;
        if (m < p.M && nb < p.N) {
          uint4 *dst = reinterpret_cast<uint4 *>(p.y + (size_t)m * p.N + nb);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (nb + 8 * g >= p.N) break;
            uint32_t o[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int j = 8 * g + 2 * h;
              float v0 = __uint_as_float(r[j]) * (sx * __ldg(p.w_scale + nb + j));
              float v1 = __uint_as_float(r[j + 1]) * (sx * __ldg(p.w_scale + nb + j + 1));
              if (p.bias) {
                v0 += bf16_bits_to_f32(__ldg(p.bias + nb + j));
                v1 += bf16_bits_to_f32(__ldg(p.bias + nb + j + 1));
              }
              o[h] = pack_bf16x2(v0, v1);
            }
            dst[g] = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    }
  }
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, QLIN_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, BN);
}

// ===================================================== W8A16 swap-AB GEMM
struct SwapParams {
  int M, N, K;
  int splits;  // CTAs per cluster along K (gridDim.z)
  const float *w_scale;
  const uint16_t *bias;
  uint16_t *y;
  unsigned *status;
};

template <int BNT>
struct SwapCfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int CONV_BYTES = BM * BK * 2;  // BF16 A tile, 128-byte swizzle
  static constexpr int X_BYTES = BNT * BK * 2;    // BF16 B tile, 128-byte swizzle
  static constexpr int RAW_BYTES = BM * BK;       // 8-bit weight tile, row-major 64 B rows
  static constexpr int STAGE_BYTES = CONV_BYTES + X_BYTES + RAW_BYTES;
  static constexpr int STAGES = (180 * 1024) / STAGE_BYTES > 8 ? 8 : (180 * 1024) / STAGE_BYTES;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr int TMEM_COLS = BNT < 32 ? 32 : BNT;
  static constexpr uint32_t IDESC = umma_idesc(1, 1, BM, BNT);
  static_assert(BM * BNT * 4 <= STAGES * STAGE_BYTES, "split-K partial tile must fit the stage ring");
};

// 16 weight codes -> 16 exact BF16 values (two 16-byte chunks, k order kept).
template <int QT>
__device__ __forceinline__ void convert16(uint4 raw, uint4 &lo, uint4 &hi) {
  uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t o[8];
  if constexpr (QT == QLIN_INT8) {
    // byte b (two's complement) -> fp32 via the 2^23 + (b ^ 0x80) bit pattern, minus 2^23 + 128: exact.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t u = w[i] ^ 0x80808080u;
      const float f0 = __uint_as_float(__byte_perm(u, 0x4Bu, 0x4550)) - 8388736.0f;
      const float f1 = __uint_as_float(__byte_perm(u, 0x4Bu, 0x4551)) - 8388736.0f;
      const float f2 = __uint_as_float(__byte_perm(u, 0x4Bu, 0x4552)) - 8388736.0f;
      const float f3 = __uint_as_float(__byte_perm(u, 0x4Bu, 0x4553)) - 8388736.0f;
      o[2 * i] = pack_bf16x2(f0, f1);
      o[2 * i + 1] = pack_bf16x2(f2, f3);
    }
  } else {
    // E4M3 pair -> f16x2 (exact) -> fp32 -> BF16 (exact: every E4M3 value is a BF16 value).
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const unsigned short pair = (unsigned short)(w[i] >> (16 * h));
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
        __half2 hv = *reinterpret_cast<__half2 *>(&h2);
        const float2 f = __half22float2(hv);
        o[2 * i + h] = pack_bf16x2(f.x, f.y);
      }
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

template <int BNT, int QT>
__global__ void __launch_bounds__(256, 1)
    k_w8_swap(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x, SwapParams p) {
  using C = SwapCfg<BNT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *full = (uint64_t *)(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t *conv_full = full + C::STAGES;
  uint64_t *empty = conv_full + C::STAGES;
  uint64_t *acc_full = empty + C::STAGES;
  uint32_t *tmem_slot = (uint32_t *)(acc_full + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * C::BM, m0 = blockIdx.y * BNT;
  const int split = blockIdx.z, S = p.splits;
  const int KB = (p.K + C::BK - 1) / C::BK;
  const int kb0 = (int)((int64_t)split * KB / S), kb1 = (int)((int64_t)(split + 1) * KB / S);
  const int nkb = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&conv_full[s], 4);
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

  if (warp == 0 && lane == 0) {  // ---------------- TMA producer
    for (int i = 0; i < nkb; ++i) {
      const int s = i % C::STAGES;
      if (i >= C::STAGES && !mbar_wait(&empty[s], ((i / C::STAGES) & 1) ^ 1, abort_flag)) {
        *abort_flag = 1;
        break;
      }
      uint8_t *st = smem + s * C::STAGE_BYTES;
      const int kx = (kb0 + i) * C::BK;
      mbar_arrive_expect_tx(&full[s], C::RAW_BYTES + C::X_BYTES);
      tma_load_2d(&tm_w, &full[s], st + C::CONV_BYTES + C::X_BYTES, kx, n0);
      tma_load_2d(&tm_x, &full[s], st + C::CONV_BYTES, kx, m0);
    }
  } else if (warp == 1 && lane == 0) {  // ---------- MMA issuer
    bool ok = true;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % C::STAGES;
      const uint32_t ph = (i / C::STAGES) & 1;
      if (!mbar_wait(&full[s], ph, abort_flag) || !mbar_wait(&conv_full[s], ph, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a = smem_u32(smem + s * C::STAGE_BYTES);
      const uint64_t ad = umma_desc_sw128(a), bd = umma_desc_sw128(a + C::CONV_BYTES);
#pragma unroll
      for (int kk = 0; kk < C::BK / 16; ++kk)  // K = 16 per instruction (32 bytes)
        mma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, C::IDESC, (i | kk) != 0);
      mma_commit(&empty[s]);
    }
    if (!ok) *abort_flag = 1;
    mma_commit(acc_full);
  } else if (warp >= 4) {  // -------------- converters, then epilogue
    const int ct = threadIdx.x - 128;  // 0..127
    bool ok = true;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % C::STAGES;
      if (!mbar_wait(&full[s], (i / C::STAGES) & 1, abort_flag)) {
        ok = false;
        break;
      }
      const uint32_t st = smem_u32(smem + s * C::STAGE_BYTES);
      const uint32_t raw = st + C::CONV_BYTES + C::X_BYTES;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = ct + 128 * j;  // 16-byte chunk of the raw tile: row r, quarter qq
        const int r = c >> 2, qq = c & 3;
        uint4 lo, hi;
        convert16<QT>(lds128(raw + r * 64 + qq * 16), lo, hi);
        const uint32_t row = st + r * 128;
        sts128(row + (((2 * qq) ^ (r & 7)) << 4), lo);
        sts128(row + (((2 * qq + 1) ^ (r & 7)) << 4), hi);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&conv_full[s]);
    }
    if (!ok) *abort_flag = 1;
    // ---- epilogue: lane = output channel n, columns = tokens
    const int q = warp & 3;
    const int nl = q * 32 + lane;
    const int n = n0 + nl;
    ok = mbar_wait(acc_full, 0, abort_flag) && ok;
    tc_fence_after();
    // tcgen05.ld is warp-collective: every lane of the warp takes the same path
    const bool run = __all_sync(0xffffffffu, ok && !*abort_flag);
    if (S == 1) {
      const bool valid = n < p.N;
      const float sw = valid ? __ldg(p.w_scale + n) : 0.0f;
      const float b = (valid && p.bias) ? bf16_bits_to_f32(__ldg(p.bias + n)) : 0.0f;
      if (run) {
#pragma unroll 1
        for (int c = 0; c < BNT; c += 16) {
          uint32_t r[16];
          tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c, r);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int m = m0 + c + j;
              if (m < p.M) p.y[(size_t)m * p.N + n] = f32_to_bf16_bits(fmaf(__uint_as_float(r[j]), sw, b));
            }
          }
        }
      }
    } else {
      // split-K: partial tile -> own shared memory, column-major [token][channel]
      float *red = reinterpret_cast<float *>(smem);
#pragma unroll 1
      for (int c = 0; c < BNT; c += 16) {
        uint32_t r[16];
        if (run) {
          tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c, r);
          tmem_ld_wait();
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) red[(c + j) * C::BM + nl] = run ? __uint_as_float(r[j]) : 0.0f;
      }
    }
  }
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, QLIN_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (S > 1) {
    cluster_sync();  // every CTA of the cluster has written its partial tile
    if (warp >= 4) {
      const int ct = threadIdx.x - 128;
      const uint32_t base = smem_u32(smem);
      constexpr int U = BNT * C::BM / 4;  // float4 units of the tile
      const int u0 = (int)((int64_t)split * U / S), u1 = (int)((int64_t)(split + 1) * U / S);
      for (int u = u0 + ct; u < u1; u += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < S; ++r) {  // fixed order: deterministic
          const uint4 v = ld_dsmem_v4(map_peer_smem(base + 16u * u, (uint32_t)r));
          acc.x += __uint_as_float(v.x);
          acc.y += __uint_as_float(v.y);
          acc.z += __uint_as_float(v.z);
          acc.w += __uint_as_float(v.w);
        }
        const int e = 4 * u, j = e / C::BM, nl = e % C::BM;
        const int m = m0 + j, n = n0 + nl;
        if (m < p.M && n < p.N) {
          float v[4] = {acc.x, acc.y, acc.z, acc.w};
          uint32_t o[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float a0 = v[2 * h] * __ldg(p.w_scale + n + 2 * h);
            float a1 = v[2 * h + 1] * __ldg(p.w_scale + n + 2 * h + 1);
            if (p.bias) {
              a0 += bf16_bits_to_f32(__ldg(p.bias + n + 2 * h));
              a1 += bf16_bits_to_f32(__ldg(p.bias + n + 2 * h + 1));
            }
            o[h] = pack_bf16x2(a0, a1);
          }
          *reinterpret_cast<uint2 *>(p.y + (size_t)m * p.N + n) = make_uint2(o[0], o[1]);
        }
      }
    }
    cluster_sync();  // no CTA leaves while a peer may still read its shared memory
  }
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ================================================================ launchers
template <class KernelT>
static cudaError_t set_smem(KernelT kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int BN>
static cudaError_t launch_fp8_bn(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st) {
  using C = Fp8Cfg<BN>;
  CUtensorMap ta, tb;
  if (!make_map(&ta, g.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.M, g.K, C::BK, C::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&tb, g.qw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.N, g.K, C::BK, BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static cudaError_t attr = set_smem(k_fp8_gemm<BN>, C::SMEM);
  if (attr != cudaSuccess) return attr;
  Fp8Params p{(int)g.M, (int)g.N, (int)g.K, g.w_scale, g.x_scale, g.bias, (uint16_t *)g.y, dev.status};
  dim3 grid((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + C::BM - 1) / C::BM));
  k_fp8_gemm<BN><<<grid, 256, C::SMEM, st>>>(ta, tb, p);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_fp8_gemm(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st) {
  if (g.M == 0) return cudaSuccess;
  if (g.N % 256 == 0 || g.N > 1024) return launch_fp8_bn<256>(g, dev, st);
  return launch_fp8_bn<128>(g, dev, st);
}

int w8_swap_bnt(int64_t M) {
  return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
}

int w8_swap_splits(int64_t M, int64_t K, int64_t N, int sms) {
  const int64_t tiles = ((N + 127) / 128) * ((M + w8_swap_bnt(M) - 1) / w8_swap_bnt(M));
  const int64_t kb = (K + 63) / 64;
  if (tiles * 4 >= (int64_t)sms * 3) return 1;
  int64_t s = sms / tiles;
  if (s > 8) s = 8;
  if (s > kb / 2) s = kb / 2;
  return s < 1 ? 1 : (int)s;
}

template <int BNT, int QT>
static cudaError_t launch_swap_t(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st) {
  using C = SwapCfg<BNT>;
  CUtensorMap tw, tx;
  if (!make_map(&tw, g.qw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.N, g.K, C::BK, C::BM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&tx, g.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.M, g.K, C::BK, BNT, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static cudaError_t attr = set_smem(k_w8_swap<BNT, QT>, C::SMEM);
  if (attr != cudaSuccess) return attr;
  const int S = w8_swap_splits(g.M, g.K, g.N, dev.sms);
  SwapParams p{(int)g.M, (int)g.N, (int)g.K, S, g.w_scale, g.bias, (uint16_t *)g.y, dev.status};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((g.N + C::BM - 1) / C::BM), (unsigned)((g.M + BNT - 1) / BNT), (unsigned)S);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 1;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = (unsigned)S;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_w8_swap<BNT, QT>, tw, tx, p);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int QT>
static cudaError_t launch_swap_q(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st) {
  switch (w8_swap_bnt(g.M)) {
    case 16: return launch_swap_t<16, QT>(g, dev, st);
    case 32: return launch_swap_t<32, QT>(g, dev, st);
    case 64: return launch_swap_t<64, QT>(g, dev, st);
    case 128: return launch_swap_t<128, QT>(g, dev, st);
    default: return launch_swap_t<256, QT>(g, dev, st);
  }
}

cudaError_t launch_w8a16_swap(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st) {
  if (g.M == 0) return cudaSuccess;
  return g.qtype == QLIN_INT8 ? launch_swap_q<QLIN_INT8>(g, dev, st) : launch_swap_q<QLIN_E4M3>(g, dev, st);
}

}  // namespace qlin
