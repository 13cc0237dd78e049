// Tensor-core (tcgen05) GEMMs for the quantized linear on sm_103a.
//
// k_fp8_gemm   W8A8 with E4M3 activations and weights.  Persistent: each CTA
//              walks 128-token x 256-channel output tiles.  TMA loads both
//              8-bit operand tiles (128-byte swizzle) into a 4-stage
//              shared-memory ring, one thread issues tcgen05.mma kind::f8f6f4
//              into one of two TMEM accumulators (fp32), and eight epilogue
//              warps read the other accumulator and apply
//              y = acc * (s_x * s_w[n]) + bias[n] -> BF16 (TMA stores).  The
//              XQ variant also quantizes the BF16 activations inside the GEMM.
//
// k_w8_dq      W8A16 (INT8 or E4M3 weight codes, BF16 activations) and the
//              INT8 W8A8 core, with the weights as the 128-row MMA operand
//              ("swap AB": output channels on the TMEM lanes, tokens on the
//              MMA N dimension, 16..256), so decode batches of a few tokens
//              still fill the tensor core's M.  TMA streams raw 8-bit weight
//              tiles and BF16 activation tiles; three converter quads turn each
//              raw tile into exact BF16 and store it into a ring of A operands
//              in tensor memory (tcgen05.st); two issuer threads alternate
//              k-blocks of tcgen05.mma kind::f16 (A from TMEM, B from shared
//              memory).  When there are too few output tiles to fill the GPU,
//              the K range is split over the CTAs of a cluster and the fp32
//              partial tiles are summed in a fixed order through distributed
//              shared memory -- one kernel, deterministic, no global workspace
//              and no spinning on global flags.
//
// Warp roles are listed at each kernel.  Every mbarrier wait is bounded
// (tc::mbar_wait); a wait that runs out sets the device status word and the CTA
// leaves through the same exit path (TMEM freed, cluster barriers met).
#include <cudaTypedefs.h>

#include <cstdlib>
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
// Persistent: each CTA walks output tiles t = blockIdx.x + j * gridDim.x
// (128 tokens x 256 channels).  TMEM holds two 256-column fp32 accumulators,
// so the epilogue of one tile overlaps the MMAs of the next.  Warps: 0 = TMA
// producer, 1 = TMEM allocator + MMA issuer, 4..11 = epilogue (two quads, each
// owning 128 of the tile's 256 channels).
struct Fp8Params {
  int M, N, K;  // N: output channels (the intermediate size I when glu)
  int mtiles, ntiles;
  int xs_per_token;  // x_scale holds one scale per token row
  int glu;           // merged gate_up: B tile = 128 gate rows + the matching 128 up rows
  // Fused static quantization (XQ): warps 2-3 of every CTA quantize the BF16
  // activations (read through tm_x) into the codes xq_dst that tm_a reads, one
  // task per (m-tile, 128-k block); a task's flag (xq_flags, row stride
  // xq_fstride) becomes 1 when all of its codes are written, and the
  // count of band b (xq_flags[mtiles * xq_fstride + b]) counts its finished tasks.  Tasks run
  // in bands of xq_band m-tiles, k-major inside a band.
  uint8_t *xq_dst;
  unsigned *xq_flags;
  int xq_fstride, xq_band;
  const float *w_scale;
  const float *x_scale;
  const uint16_t *bias;
  uint16_t *y;
  unsigned *status;
};

// XQ roles of the 512-thread variant: warp 2 stages BF16 chunks (TMA), warps
// 12..15 convert them, warp 3 publishes finished tasks.
constexpr int kXqConverters = 4;
constexpr int kXqPrefetch = 0;  // chunks brought into L2 ahead of the staging ring

// GEMM pipeline depth of the fused-quantization variant (CTA pairs, 32 KB
// stages): 4 stages, the output staging and 3 chunks of activation staging.
constexpr int kFp8XqStages = 4;

// PAIR = 1: the two CTAs of a 2-CTA cluster compute a 256 x 256 tile with
// pair MMAs (cta_group::2): each CTA stages its own 128 tokens of A and 128 of
// the 256 channels of B, so a stage is 32 KB instead of 48 KB, and the MMA
// reads each CTA's B half once for both CTAs' rows.
template <int XQ, int PAIR = 0>
struct Fp8CfgT {
  static constexpr int BM = 128, BN = 256, BK = 128, STAGES = XQ ? kFp8XqStages : PAIR ? 6 : 4;
  static constexpr int A_BYTES = BM * BK, B_BYTES = (PAIR ? BN / 2 : BN) * BK, STAGE_BYTES = A_BYTES + B_BYTES;
  // epilogue: two 32 x 32 BF16 blocks per epilogue warp, staged for TMA stores
  // (one fills while the other's store reads it)
  static constexpr int EPI_OFF = STAGES * STAGE_BYTES, EPI_WARP_BYTES = 32 * 32 * 2;
  static constexpr int EPI_BYTES = 8 * 2 * EPI_WARP_BYTES;
  // XQ: a ring of chunks (XQ_ROWS rows of a task's 128 x 128 BF16 activation
  // tile), TMA-staged, as many as the rest of the shared memory holds
  static constexpr int XQ_ROWS = 64, XQ_CPT = BM / XQ_ROWS, XQ_CHUNK = XQ_ROWS * BK * 2;
  static constexpr int XQ_OFF = EPI_OFF + EPI_BYTES;
  static constexpr int XQ_NBUF = XQ ? (227 * 1024 - XQ_OFF - 256 - 1024) / XQ_CHUNK : 0;
  static_assert(XQ == 0 || PAIR == 1, "the fused-quantization variant runs CTA pairs (32 KB stages)");
  static constexpr int BAR_OFF = XQ_OFF + XQ_NBUF * XQ_CHUNK;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;
  static constexpr int THREADS = XQ ? 512 : 384;
  static constexpr uint32_t IDESC = umma_idesc(0, 0, PAIR ? 2 * BM : BM, BN);
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(XQ == 0 || (XQ_NBUF >= 2 && XQ_NBUF <= 6), "chunk ring (barriers and counters at BAR_OFF + 128)");
};
using Fp8Cfg = Fp8CfgT<0>;

// XQ = 1: the activations are quantized inside the kernel.  Warps 2-3 and
// 12-15 (a 512-thread block) of every CTA take quantization tasks (m-tile,
// 128-k block).  TMA streams each task's BF16 tile into a ring of 64-row chunks
// in shared memory, several tasks ahead; the warps write the E4M3 codes to
// global memory and release the task's flag and its band's count.  Tasks go in
// bands of m-tiles about one wave of GEMM tiles wide, k-major inside a band, so
// the first k-blocks of every tile of a wave are ready first.  The TMA producer
// loads a tile with no checks once it has seen the tile's band (and all before
// it) complete; otherwise it acquires a group of four task flags (the next
// group's load already in flight) before loading those A tiles, and fences the
// async proxy after either acquire.  The quantization streams from HBM while
// the GEMM is bound by the tensor cores and L2, so it overlaps.  The launch is
// cooperative: every CTA is resident, and every wait is bounded besides.
//
// PAIR = 1 (2-CTA clusters): work items are pair tiles, 256 tokens (m-tiles 2q
// and 2q + 1, one per CTA) by 256 channels (128 per CTA).  Only the even CTA
// issues MMAs.  Both CTAs' TMA loads count their bytes on the even CTA's full
// barrier; the MMA commits arrive on the empty and accumulator barriers of both
// CTAs; both CTAs' epilogue warps release an accumulator on the even CTA's
// barrier.  Each CTA's tensor memory holds its own 128 tokens of the tile.
template <int XQ, int PAIR>
__global__ void __launch_bounds__(Fp8CfgT<XQ, PAIR>::THREADS, 1)
    k_fp8_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y, Fp8Params p) {
  using C = Fp8CfgT<XQ, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint64_t *full = (uint64_t *)(smem + C::BAR_OFF);
  uint64_t *empty = full + C::STAGES;
  uint64_t *acc_full = empty + C::STAGES, *acc_empty = acc_full + 2;
  uint32_t *tmem_slot = (uint32_t *)(acc_empty + 2);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (p.K + C::BK - 1) / C::BK;
  if constexpr (PAIR) {
    // Launched without its 2-CTA cluster shape, the pair MMAs, loads and barrier
    // arrivals would address a CTA that does not exist: report and leave before
    // any barrier, tensor memory or peer is touched.
    if (cluster_nctarank() != 2) {
      if (threadIdx.x == 0) set_status(p.status, QLIN_ERR_UNSUPPORTED);
      return;
    }
  }
  const int rank = PAIR ? (int)(cluster_ctarank() & 1u) : 0;
  // work items t = cid + j * G, m-group major: output tiles, or pair tiles
  // (m-tiles 2q, 2q + 1 of one n-tile)
  const int mgroups = PAIR ? (p.mtiles + 1) / 2 : p.mtiles;
  const int items = mgroups * p.ntiles, G = gridDim.x / (PAIR + 1), cid = blockIdx.x / (PAIR + 1);
  const int my_tiles = (cid < items) ? (items - cid + G - 1) / G : 0;
  auto tile_m0 = [&](int t) { return ((t / p.ntiles) * (PAIR + 1) + rank) * C::BM; };
  auto tile_n0 = [&](int t) { return (t % p.ntiles) * C::BN; };
  // the even CTA's barrier at the same offset as `bar` (shared::cluster address)
  auto leader = [&](uint64_t *bar) { return PAIR ? map_peer_smem(smem_u32(bar), 0) : smem_u32(bar); };
  auto peer = [&](uint64_t *bar) { return map_peer_smem(smem_u32(bar), 1); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // the MMA commit that has read the stage
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], PAIR ? 16 : 8);  // the epilogue warps (of both CTAs of a pair)
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_y);
    if constexpr (XQ == 1) {
      uint64_t *xq_full = (uint64_t *)(smem + C::BAR_OFF + 128), *xq_empty = xq_full + C::XQ_NBUF;
      unsigned *xq_count = (unsigned *)(xq_empty + C::XQ_NBUF);
      for (int b = 0; b < C::XQ_NBUF; ++b) {
        mbar_init(&xq_full[b], 1);
        mbar_init(&xq_empty[b], kXqConverters);
      }
      for (int w = 0; w < kXqConverters; ++w) xq_count[w] = 0;
      tma_prefetch_desc(&tm_x);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) tmem_alloc_pair(tmem_slot, 512);
    else tmem_alloc(tmem_slot, 512);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool pair_ok = true;
  if constexpr (PAIR) {
    cluster_sync();  // both CTAs' barriers exist before a load, commit or arrival reaches them
    // both CTAs must hold the same tensor-memory address; otherwise neither does any work
    pair_ok = ld_dsmem_u32(map_peer_smem(smem_u32(tmem_slot), (uint32_t)(rank ^ 1))) == tmem;
    if (!pair_ok && threadIdx.x == 0) set_status(p.status, QLIN_ERR_UNSUPPORTED);
  }
  pdl_wait();  // inputs of the previous kernel in the stream are complete from here on
  pdl_trigger();

  if (!pair_ok) {
    // a pair whose tensor memory does not match does nothing but leave together
  } else if (warp == 0) {  // ------------------------------- TMA producer
    if (lane == 0) {
      int i = 0;
      // XQ: the tiles of bands 0..ready_band (seen complete, fenced once) load
      // with no flag checks; the others check the flags of each group of four
      // k-blocks, the next group's flags loaded one group ahead.
      auto group_flags = [&](int t, int g) { return p.xq_flags + (tile_m0(t) / C::BM) * p.xq_fstride + 4 * g; };
      const unsigned *band_done = p.xq_flags + p.mtiles * p.xq_fstride;
      int ready_band = -1;
      uint4 pf = make_uint4(0, 0, 0, 0);
      for (int j = 0; j < my_tiles && !*abort_flag; ++j) {
        const int t = cid + j * G;
        const int m0 = tile_m0(t), n0 = tile_n0(t);
        bool tile_ready = true;
        if constexpr (XQ == 1) {
          const int band = (m0 / C::BM) / p.xq_band;
          if (m0 < p.M && band > ready_band) {
            pf = ld_relaxed_v4(group_flags(t, 0));  // in flight while the band counters are read
            int b = ready_band + 1;
            while (b <= band &&
                   ld_relaxed_u32(band_done + b) >= (unsigned)(min(p.xq_band, p.mtiles - b * p.xq_band) * nkb))
              ++b;
            if (b > ready_band + 1) {
              fence_acq_rel_gpu();         // acquire: every code of those bands is written
              fence_proxy_async_global();  // ... before this thread's TMA reads of them
              ready_band = b - 1;
            }
            tile_ready = band <= ready_band;
          }
        }
        for (int kb = 0; kb < nkb; ++kb, ++i) {
          const int s = i % C::STAGES;
          if constexpr (XQ == 1) {
            if (!tile_ready && (kb & 3) == 0) {
              uint4 cur = pf;
              if (kb + 4 < nkb) pf = ld_relaxed_v4(group_flags(t, kb / 4 + 1));  // the next group
              const int need = min(4, nkb - kb);  // flags of k-blocks past K are never set
              auto ready = [&](uint4 v) {
                return v.x != 0u && (need < 2 || v.y != 0u) && (need < 3 || v.z != 0u) && (need < 4 || v.w != 0u);
              };
              if (!ready(cur)) {
                const uint64_t t0 = globaltimer_ns();
                while (!ready(cur = ld_relaxed_v4(group_flags(t, kb / 4)))) {
                  if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
                    *abort_flag = 1;
                    break;
                  }
                  __nanosleep(64);
                }
                if (*abort_flag) break;
              }
              fence_acq_rel_gpu();         // acquire: the task's code writes happen before what follows
              fence_proxy_async_global();  // ... including this thread's TMA reads of them
            }
          }
          if (i >= C::STAGES && !mbar_wait(&empty[s], ((i / C::STAGES) & 1) ^ 1, abort_flag)) {
            *abort_flag = 1;
            break;
          }
          uint8_t *st = smem + s * C::STAGE_BYTES;
          // B: two boxes of 128 rows; glu: the gate rows n0/2.. and the matching up rows N + n0/2..
          const int b0 = p.glu ? n0 / 2 : n0, b1 = p.glu ? p.N + n0 / 2 : n0 + C::BN / 2;
          if constexpr (PAIR) {  // this CTA's A tile and its B box; both CTAs' bytes count on the even CTA
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE_BYTES);
            const uint32_t fb = leader(&full[s]);
            tma_load_2d_pair(&tm_a, fb, st, kb * C::BK, m0);
            tma_load_2d_pair(&tm_b, fb, st + C::A_BYTES, kb * C::BK, rank ? b1 : b0);
          } else {
            mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
            tma_load_2d(&tm_a, &full[s], st, kb * C::BK, m0);
            tma_load_2d(&tm_b, &full[s], st + C::A_BYTES, kb * C::BK, b0);
            tma_load_2d(&tm_b, &full[s], st + C::A_BYTES + C::B_BYTES / 2, kb * C::BK, b1);
          }
        }
      }
      if constexpr (PAIR) {
        // the last stages this CTA loaded have been read by the pair's MMAs (the
        // empty barriers the MMA commits arrive on) before it leaves
        for (int k = i > C::STAGES ? i - C::STAGES : 0; k < i; ++k)
          mbar_wait_drain(&empty[k % C::STAGES], (uint32_t)(k / C::STAGES) & 1);
      } else if (*abort_flag) {
        drain_ring(full, C::STAGES, i, C::STAGES);  // abort: the stages this CTA armed land before it leaves
      }
    }
  } else if (XQ == 1 && (warp == 2 || warp == 3 || warp >= 12)) {  // ----- activation quantizer
    uint64_t *xq_full = (uint64_t *)(smem + C::BAR_OFF + 128), *xq_empty = xq_full + C::XQ_NBUF;
    unsigned *xq_count = (unsigned *)(xq_empty + C::XQ_NBUF);  // tasks finished, per converter warp
    const uint8_t *xq_buf = smem + C::XQ_OFF;
    const int tasks = p.mtiles * nkb, per_band = p.xq_band * nkb;
    const int mine = (int)blockIdx.x < tasks ? (tasks - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    auto task_of = [&](int j, int &mt, int &kb) {
      const int u = (int)blockIdx.x + j * (int)gridDim.x, band = u / per_band, r = u - band * per_band;
      const int nb = min(p.xq_band, p.mtiles - band * p.xq_band);  // the last band may be narrower
      kb = r / nb;
      mt = band * p.xq_band + (r - kb * nb);
    };
    // chunk c = part c % CPT (XQ_ROWS rows) of task c / CPT goes through ring buffer c % NB
    constexpr int NB = C::XQ_NBUF, CPT = C::XQ_CPT;
    const int chunks = CPT * mine;
    if (warp == 2) {  // ---- staging: TMA loads of BF16 chunks into the ring
      if (lane == 0) {
        // chunks kXqPrefetch ahead of the one being loaded are brought into L2,
        // so the ring's loads see L2 latency rather than HBM latency
        auto prefetch = [&](int c) {
          if (c >= chunks) return;
          int mt, kb;
          task_of(c / CPT, mt, kb);
          tma_prefetch_l2_2d(&tm_x, kb * C::BK, mt * C::BM + (c % CPT) * C::XQ_ROWS);
        };
        for (int c = 0; c < kXqPrefetch; ++c) prefetch(c);
        // the BF16 activations are read once: they must not push the GEMM's
        // reused weight and code tiles out of L2
        const uint64_t policy = l2_policy_evict_first();
        int issued = 0;
        bool ok = true;
        for (; issued < chunks; ++issued) {
          const int c = issued, b = c % NB;
          if constexpr (kXqPrefetch > 0) prefetch(c + kXqPrefetch);
          if (c >= NB && !mbar_wait(&xq_empty[b], (uint32_t)(c / NB - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          int mt, kb;
          task_of(c / CPT, mt, kb);
          mbar_arrive_expect_tx(&xq_full[b], C::XQ_CHUNK);
          tma_load_2d_hint(&tm_x, &xq_full[b], (void *)(xq_buf + b * C::XQ_CHUNK), kb * C::BK,
                           mt * C::BM + (c % CPT) * C::XQ_ROWS, policy);
        }
        if (!ok) {
          *abort_flag = 1;
          // loads that may still be in flight land before the CTA leaves
          for (int c = max(0, issued - NB); c < issued; ++c)
            mbar_wait_drain(&xq_full[c % NB], (uint32_t)(c / NB) & 1);
        }
      }
    } else if (warp == 3) {  // ---- publishing: flags and band counts of finished tasks
      if (lane == 0) {
        int released = 0;
        while (released < mine) {
          int done = 0;
          const uint64_t t0 = globaltimer_ns();
          while (true) {
            done = mine;
            for (int w = 0; w < kXqConverters; ++w) done = min(done, (int)ld_acquire_cta_shared(&xq_count[w]));
            if (done > released || *abort_flag) break;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
              *abort_flag = 1;
              break;
            }
            __nanosleep(32);
          }
          if (done <= released) break;  // aborted
          // one release for every task finished since the last: the acquire
          // loads above saw all their code stores, and the fence is cumulative
          fence_proxy_async_global();  // the codes are read through the async proxy (TMA)
          fence_acq_rel_gpu();
          for (; released < done; ++released) {
            int mt, kb;
            task_of(released, mt, kb);
            red_relaxed_add_u32(p.xq_flags + mt * p.xq_fstride + kb, 1u);
            red_relaxed_add_u32(p.xq_flags + p.mtiles * p.xq_fstride + mt / p.xq_band, 1u);
          }
        }
      }
    } else {  // ---- conversion: warps 12..15, 128 threads
      const int qt = threadIdx.x - 384;
      const StaticE4m3 xs = make_static_e4m3(__ldg(p.x_scale));
      for (int c = 0; c < chunks; ++c) {
        const int b = c % NB;
        // the warp takes one path whatever each lane's bounded wait saw
        if (!__all_sync(0xffffffffu, mbar_wait(&xq_full[b], (uint32_t)(c / NB) & 1, abort_flag))) {
          *abort_flag = 1;
          break;
        }
        int mt, kb;
        task_of(c / CPT, mt, kb);
        const uint32_t src = smem_u32(xq_buf + b * C::XQ_CHUNK);
        const int mh = mt * C::BM + (c % CPT) * C::XQ_ROWS, k0 = kb * C::BK;
        // XQ_ROWS rows x 16 pieces of 8 BF16 (16 consecutive threads cover one
        // row's 256 bytes): each thread reads its pieces first, then converts and
        // stores them, independent chains
        constexpr int PIECES = C::XQ_ROWS * 16 / (32 * kXqConverters);
        static_assert(PIECES * 32 * kXqConverters == C::XQ_ROWS * 16, "pieces per converter thread");
        uint4 v[PIECES];
#pragma unroll
        for (int i = 0; i < PIECES; ++i) v[i] = lds128(src + 16u * (qt + i * 32 * kXqConverters));
        uint2 q[PIECES];
        if (xs.c.fast) {  // uniform: the branch stays outside the unrolled conversions
#pragma unroll
          for (int i = 0; i < PIECES; ++i)
            q[i] = make_uint2(e4m3_static4_fast(v[i].x, v[i].y, xs), e4m3_static4_fast(v[i].z, v[i].w, xs));
        } else {
#pragma unroll
          for (int i = 0; i < PIECES; ++i)
            q[i] = make_uint2(e4m3_static4_exact_div(v[i].x, v[i].y, xs.c),
                              e4m3_static4_exact_div(v[i].z, v[i].w, xs.c));
        }
#pragma unroll
        for (int i = 0; i < PIECES; ++i) {
          const int e = qt + i * 32 * kXqConverters, row = e >> 4, col = k0 + (e & 15) * 8;
          if (mh + row < p.M && col < p.K) *reinterpret_cast<uint2 *>(p.xq_dst + (size_t)(mh + row) * p.K + col) = q[i];
        }
        __syncwarp();  // the warp's reads of the buffer and its code stores come before ...
        if (lane == 0) {
          mbar_arrive(&xq_empty[b]);                                             // ... the refill
          if (c % CPT == CPT - 1) red_release_cta_shared_add(&xq_count[warp - 12], 1u);  // ... the publication
        }
      }
    }
  } else if (warp == 1) {  // ------------------------ MMA issuer (the even CTA of a pair)
    if (lane == 0 && rank == 0) {
      bool ok = true;
      int i = 0;
      for (int j = 0; j < my_tiles && ok; ++j) {
        const int b = j & 1;
        if (j >= 2 && !mbar_wait(&acc_empty[b], ((j >> 1) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem + b * C::BN;
        for (int kb = 0; kb < nkb; ++kb, ++i) {
          const int s = i % C::STAGES;
          if (!mbar_wait(&full[s], (i / C::STAGES) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + s * C::STAGE_BYTES);
          const uint64_t ad = umma_desc_sw128(a), bd = umma_desc_sw128(a + C::A_BYTES);
          if constexpr (PAIR) {
            mma_fp8_pair(dt, ad, bd, C::IDESC, kb > 0 ? 1u : 0u);  // K = 32 per instruction (32 bytes)
            mma_fp8_pair(dt, ad + 2, bd + 2, C::IDESC, 1u);
            mma_fp8_pair(dt, ad + 4, bd + 4, C::IDESC, 1u);
            mma_fp8_pair(dt, ad + 6, bd + 6, C::IDESC, 1u);
            mma_commit_pair(smem_u32(&empty[s]));
            mma_commit_pair(peer(&empty[s]));
          } else {
            mma_fp8(dt, ad, bd, C::IDESC, kb > 0 ? 1u : 0u);  // K = 32 per instruction (32 bytes)
            mma_fp8(dt, ad + 2, bd + 2, C::IDESC, 1u);
            mma_fp8(dt, ad + 4, bd + 4, C::IDESC, 1u);
            mma_fp8(dt, ad + 6, bd + 6, C::IDESC, 1u);
            mma_commit(&empty[s]);
          }
        }
        if (!ok) break;
        if constexpr (PAIR) {
          mma_commit_pair(smem_u32(&acc_full[b]));
          mma_commit_pair(peer(&acc_full[b]));
        } else {
          mma_commit(&acc_full[b]);
        }
      }
      // Drain: no commit arrival may still be in flight towards this CTA's shared
      // memory when it exits (a successor CTA on this SM may already own it); the
      // wait holds on the abort path too
      if (i > 0) ok = mbar_wait_drain(&empty[(i - 1) % C::STAGES], ((i - 1) / C::STAGES) & 1) && ok;
      if (!ok) *abort_flag = 1;
    }
  } else if (warp >= 4) {  // ------------------------- epilogue
    const int q4 = warp & 3, half = (warp - 4) >> 2;  // half h owns channels [128h, 128h + 128)
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const float sx = p.xs_per_token ? 1.0f : __ldg(p.x_scale);
    // Output path: each 32 x 32 block of BF16 results (row = lane) is written into
    // one of this warp's two staging blocks with the 64-byte swizzle (16-byte chunk
    // q of row r at chunk q ^ ((r >> 1) & 3): the lanes' row writes hit distinct
    // banks), then stored by TMA, which writes whole row segments and clips rows
    // and columns outside y.  The blocks alternate, so a block is rewritten only
    // once the store issued two blocks earlier has read it.
    uint8_t *stage = smem + C::EPI_OFF + (warp - 4) * 2 * C::EPI_WARP_BYTES;
    const uint32_t sw = (lane >> 1) & 3;
    int emitted = 0;  // stores lane 0 has issued
    auto emit = [&](const uint32_t (&o)[16], int x, int y) {
      uint8_t *blk = stage + (emitted & 1) * C::EPI_WARP_BYTES;
      if (emitted >= 2) {
        if (lane == 0) bulk_wait_read_1();  // the store from two blocks ago has read this block
        __syncwarp();
      }
      const uint32_t st_row = smem_u32(blk) + 64u * lane;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        sts128(st_row + (((uint32_t)q ^ sw) << 4), make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]));
      fence_proxy_async_smem();  // the TMA store reads the block through the async proxy
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&tm_y, blk, x, y);
        bulk_commit();
      }
      ++emitted;
    };
    // Column factors of this warp's 128 columns of a tile, one float4 per lane:
    // s_x * s_w[n] and the bias, zero from channel `end` on (n is a multiple of 4
    // and end of 16, so a lane's 4 are all inside or all outside).  Plain: lane l
    // holds the tile's columns 128 half + 4l..; glu: lanes 0..15 the gate
    // channels 64 half + 4l.. (end N), lanes 16..31 their up channels N further
    // on (end 2N).  They are loaded before the wait for the tile's accumulator,
    // so their latency hides behind the MMAs; a column's factor is then one
    // shuffle from the lane that holds it.
    auto load_factors = [&](int n0, float4 &fs, float4 &fb) {
      int n = n0 + 128 * half + 4 * lane, end = p.N;
      if (p.glu) {
        const int g = n0 / 2 + 64 * half + 4 * (lane & 15);
        n = lane < 16 ? g : p.N + g;
        end = lane < 16 ? p.N : 2 * p.N;
      }
      fs = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      fb = fs;
      if (n < end) {
        const float4 w = __ldg(reinterpret_cast<const float4 *>(p.w_scale + n));
        fs = make_float4(sx * w.x, sx * w.y, sx * w.z, sx * w.w);
        if (p.bias) {
          const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p.bias + n));
          fb = make_float4(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16), bf16_bits_to_f32(v.y & 0xFFFFu),
                           bf16_bits_to_f32(v.y >> 16));
        }
      }
    };
    // component k (0..3, known at compile time) of lane src's float4, to every lane
    auto shfl4 = [&](const float4 &f, int k, int src) {
      return __shfl_sync(0xffffffffu, k == 0 ? f.x : k == 1 ? f.y : k == 2 ? f.z : f.w, src);
    };
    bool ok = true;
    for (int j = 0; j < my_tiles && ok; ++j) {
      const int t = cid + j * G, b = j & 1;
      const int m0 = tile_m0(t), n0 = tile_n0(t);
      float4 fs, fb;
      load_factors(n0, fs, fb);
      ok = mbar_wait(&acc_full[b], (j >> 1) & 1, abort_flag);
      tc_fence_after();
      // tcgen05.ld is warp-collective: every lane of the warp takes the same path
      if (!__all_sync(0xffffffffu, ok && !*abort_flag)) {
        ok = false;
        break;
      }
      const int m = m0 + q4 * 32 + lane, yrow0 = m0 + q4 * 32;
      // the second m-tile of a pair past M has no rows to write (its loads read zeros)
      if (m0 >= p.M) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR && rank) mbar_arrive_cluster(leader(&acc_empty[b]));
          else mbar_arrive(&acc_empty[b]);
        }
        continue;
      }
      // per-token activation scale multiplies the row (lane = token)
      const float sxm = p.xs_per_token ? (m < p.M ? __ldg(p.x_scale + m) : 0.0f) : 1.0f;
      if (p.glu) {
        // columns [0,128) hold gate channels n0/2 + c, columns [128,256) the matching up
        // channels; half h takes gate columns [64h, 64h + 64) and their up partners
        const int nb0 = n0 / 2;
#pragma unroll 1
        for (int c = 64 * half; c < 64 * half + 64; c += 32) {
          const int nb = nb0 + c;
          uint32_t o[16];
#pragma unroll
          for (int q = 0; q < 2; ++q) {  // 16 gate columns and their 16 up columns at a time
            uint32_t rg[16], ru[16];
            tmem_ld16(tmem + lane_base + b * C::BN + c + 16 * q, rg);
            tmem_ld16(tmem + lane_base + b * C::BN + 128 + c + 16 * q, ru);
            tmem_ld_wait();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              // gate channels nb + 16q + 8hh.. (this warp's gate column jg..), and the
              // up channels N further on, held by lanes 16..31
              const int jg = (c - 64 * half) + 16 * q + 8 * hh;
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                float v[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int i = 2 * h + e, col = 8 * hh + i, src = (jg + i) >> 2;
                  const float g = fmaf(__uint_as_float(rg[col]), sxm * shfl4(fs, i & 3, src), shfl4(fb, i & 3, src));
                  const float u =
                      fmaf(__uint_as_float(ru[col]), sxm * shfl4(fs, i & 3, 16 + src), shfl4(fb, i & 3, 16 + src));
                  v[e] = silu_f(g) * u;
                }
                o[8 * q + 4 * hh + h] = pack_bf16x2(v[0], v[1]);
              }
            }
          }
          emit(o, nb, yrow0);
        }
      } else {
#pragma unroll 1
        for (int c = 128 * half; c < 128 * half + 128; c += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + b * C::BN + c, r);
          const int nb = n0 + c;
          tmem_ld_wait();
          uint32_t o[16];
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              // this warp's columns j, j + 1 (j even): factors from lane j / 4
              const int i = 2 * h, col = 8 * hh + i, j = (c - 128 * half) + col, src = j >> 2;
              o[4 * hh + h] = pack_bf16x2(
                  fmaf(__uint_as_float(r[col]), sxm * shfl4(fs, i & 3, src), shfl4(fb, i & 3, src)),
                  fmaf(__uint_as_float(r[col + 1]), sxm * shfl4(fs, (i + 1) & 3, src), shfl4(fb, (i + 1) & 3, src)));
            }
          }
          if (nb < p.N) emit(o, nb, yrow0);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && rank) mbar_arrive_cluster(leader(&acc_empty[b]));
        else mbar_arrive(&acc_empty[b]);
      }
    }
    // every store has written y (and read its staging block) before the CTA leaves
    if (lane == 0 && emitted > 0) bulk_wait_all();
    __syncwarp();
    if (!ok) *abort_flag = 1;
  }
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, QLIN_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (PAIR) {
    // neither CTA frees the pair's tensor memory or leaves while the other may
    // still send it loads, commits or arrivals (every wait above is bounded, so
    // both get here); on the abort path what was sent is given time to land
    cluster_sync();
    if (*abort_flag) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
    }
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
  } else {
    if (warp == 1) tmem_dealloc(tmem, 512);
  }
}

// ========================================== swap-AB GEMM with A in tensor memory
// Output channels on the 128 TMEM lanes, tokens on the MMA N dimension (16..256).
// The 8-bit weight codes stream through a deep shared-memory ring; converter
// warps turn each 128 x 64 tile into exact BF16 and store it straight into a
// ring of A operands in tensor memory (tcgen05.st), so the converted weights
// never touch shared memory; the MMA reads A from TMEM and the activations (B)
// from a 128-byte-swizzled shared-memory ring.
//
// Modes:  W8A16: B = BF16 activations, fp32 accumulation over all of K,
//                epilogue y = acc * s_w[n] + bias[n].
//         I8 fused: B = raw BF16 activations; the converter quad that takes a
//                k-block also quantizes that block's activation tile in place
//                (static per-tensor scale) into integer-valued BF16 before it
//                releases the block to the MMA, so the linear is one kernel.
//         I8:    B = activation codes stored as integer-valued BF16; the MMA
//                accumulates fp32 over chunks of 1024 k, where every partial sum
//                is an integer below 127*127*1024 < 2^24 and therefore exact; the
//                epilogue warps add each chunk into int32 sums (registers, or
//                tensor memory for 128-token tiles), so the full accumulator is
//                the exact integer sum.  Output: raw int32, or
//                y = acc * (s_x * s_w[n]) + bias[n].
enum SwapMode { kSwapW8A16 = 0, kSwapI8Scaled = 1, kSwapI8Raw = 2, kSwapI8Fused = 3 };

struct SwapParams {
  int M, N, K;       // N: output channels (the intermediate size I when glu)
  int xs_per_token;  // x_scale holds one scale per token (I8 scaled mode)
  int glu;           // merged gate_up: a 128-row tile = 64 gate rows + their 64 up rows
  int splits;        // CTAs per cluster along K (gridDim.z)
  int units;   // output tiles: n-tiles x token tiles
  int ntiles;  // n-tiles (128 channels each)
  const float *w_scale;
  const float *x_scale;
  const uint16_t *bias;
  void *y;
  unsigned *status;
};

template <int BNT, int MODE = 0>
struct DqCfg {
  static constexpr int BM = 128, BK = 64;
  static constexpr int RAW_BYTES = BM * BK;     // 8-bit weight tile, 64-byte swizzle
  static constexpr int X_BYTES = BNT * BK * 2;  // BF16 activation tile, 128-byte swizzle
  static constexpr int QUADS = 3;               // converter warp quads
  static constexpr int THREADS = 640;           // 20 warps
  // Accumulators.  A chain of MMAs into one small tile is bound by the MMA's
  // accumulate latency, not its throughput, so consecutive k-blocks rotate
  // over NACC independent accumulator tiles (summed in a fixed order by the
  // epilogue); ND sets of them alternate between consecutive output tiles.
  // INT8 (exact int32 sums) with 128-token tiles: the epilogue's running int32
  // sums live in tensor memory (SUMCOL..SUMCOL + BNT) instead of registers, one
  // accumulator per chunk, two alternating.
  static constexpr bool TSUM = MODE != 0 && BNT > 64;
  static constexpr int NACC = TSUM ? 1 : BNT <= 32 ? 4 : BNT <= 128 ? 2 : 1;
  static constexpr int ISSUERS = NACC >= 2 ? 2 : 1;  // MMA-issuing threads (own accumulators each)
  static constexpr int DSTRIDE = NACC * BNT;         // columns of one accumulator set
  static constexpr int ND = TSUM || 2 * DSTRIDE <= 256 ? 2 : 1;
  static constexpr int SUMCOL = ND * DSTRIDE;  // TSUM: int32 running sums
  // first TMEM column of the A ring
  static constexpr int ACOL = TSUM ? SUMCOL + BNT : ND * DSTRIDE <= 128 ? 128 : 256;
  // Ring depths.  mbarrier.try_wait.parity only tells the current phase from
  // the previous one, so a waiter must never be more than one phase ahead of a
  // slot.  Every waiter below is one of several consumers that take blocks
  // round-robin; it is safe when the previous use of its slot was its own
  // earlier block, i.e. when the ring depth is a multiple of the number of
  // consumers sharing that ring:
  //   raw ring      (3 converter quads)               R  % 3 == 0
  //   TMEM A ring   (3 quads wait a_empty, issuers     NA % (3 x ISSUERS) == 0
  //                  wait a_full)
  //   activations   (QX: the 3 quads wait x_full)      X  % 3 == 0
  // An issuer waits on one barrier per block, a_full, which completes only once
  // both the block's converted weights are in tensor memory and its
  // activation tile has landed:
  //   XA (X <= NA, no in-place quantization): the activation tile's TMA
  //      completes on the block's a_full itself (one more arrival, with its
  //      bytes).  The load of block i follows the MMA of block i - X, so the
  //      issuers have consumed a_full's previous phase (block i - NA) by then.
  //   QX: the converter quad waits for the tile (x_full) before it arrives.
  // 256-token tiles keep four 32 KB activation stages (three were slower).
  static constexpr int NA = TSUM ? 3 : ACOL == 128 ? 12 : 6;  // A stages, 32 columns (64 BF16 k) each
  static constexpr int X = MODE == 3 ? (BNT <= 32 ? 18 : 12) : BNT <= 32 ? 18 : BNT == 64 ? 9 : BNT == 128 ? 6 : 4;
  static constexpr bool XA = MODE != 3 && X <= NA;
  static constexpr bool QX = !XA;
  static constexpr int RING = 200 * 1024;
  static constexpr int R0 = (RING - X * X_BYTES) / RAW_BYTES;
  static constexpr int R = (R0 > 15 ? 15 : R0) / 3 * 3;  // raw stages
  static constexpr int X_OFF = 0, RAW_OFF = X * X_BYTES, BAR_OFF = RAW_OFF + R * RAW_BYTES;
  // merged gate_up: per 16-token chunk the gate rows pass g of tokens 8..15 and the up
  // rows u of tokens 0..7 to each other; two slots, so a side can run one chunk ahead
  static constexpr int XCHG_OFF = BAR_OFF + 1024, XCHG_BYTES = 2 * 2 * 8 * 64 * 4;
  // split-K: the tile's per-row weight scales and biases and per-token scales,
  // staged while the main loop runs
  static constexpr int SCL_OFF = XCHG_OFF + XCHG_BYTES, SCL_BYTES = (2 * BM + BNT) * 4;
  static constexpr int SMEM = SCL_OFF + SCL_BYTES + 1024;  // + alignment slack
  static constexpr uint32_t IDESC = umma_idesc(1, 1, BM, BNT);
  static_assert(R % QUADS == 0 && R >= 6, "raw ring depth: multiple of the converter quads");
  static_assert(NA % (QUADS * ISSUERS) == 0, "A ring depth: multiple of quads x issuers");
  static_assert(XA || X % QUADS == 0, "activation ring depth: multiple of the quads that wait on it");
  static_assert(ND * DSTRIDE <= ACOL && ACOL + NA * 32 <= 512, "TMEM columns");
  static_assert(BM * BNT * 4 <= BAR_OFF, "split-K partial tile must fit the rings");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(2 * (R + X + NA + ND + 4) * 8 + 16 <= 1024, "barrier area");
};

// 16 weight codes -> 16 exact BF16 values packed in 8 words (k order kept).
template <int QT>
__device__ __forceinline__ void convert16(uint4 raw, uint32_t *o) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  if constexpr (QT == QLIN_INT8) {
    // byte b (two's complement) -> fp32 via the 2^23 + (b ^ 0x80) bit pattern, minus 2^23 + 128: exact.
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t u = w[i] ^ 0x80808080u;
      const float f0 = __uint_as_float(__byte_perm(u, 0x4Bu, 0x4550)) - 8388736.0f;
      const float f1 = __uint_as_float(__byte_perm(u, 0x4Bu, 0x4551)) - 8388736.0f;
      const float f2 = __uint_as_float(__byte_perm(u, 0x4Bu, 0x4552)) - 8388736.0f;
      const float f3 = __uint_as_float(__byte_perm(u, 0x4Bu, 0x4553)) - 8388736.0f;
      o[2 * i] = pack_code_bf16x2(f0, f1);
      o[2 * i + 1] = pack_code_bf16x2(f2, f3);
    }
  } else {
    // E4M3 code s.eeee.mmm -> BF16 with the sign at bit 15 and eeee.mmm at bits
    // 4..10: that BF16 number is the code's value times 2^-120 (a normal code has
    // BF16 exponent field eeee and mantissa mmm/8; a subnormal code 0.mmm * 2^-6
    // becomes the BF16 subnormal mmm * 2^-129), so one exact BF16 multiply by
    // 2^120 gives the value.  Integer and FMA-pipe instructions only.
    const __nv_bfloat162 k2p120 = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)0x7B80),
                                                     __ushort_as_bfloat16((unsigned short)0x7B80));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // codes 2h, 2h+1 of the word into the high bytes of the two 16-bit halves
        const uint32_t t = __byte_perm(w[i], 0u, h ? 0x3424u : 0x1404u);
        const uint32_t b = ((t >> 4) & 0x07F007F0u) | (t & 0x80008000u);
        const __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&b), k2p120);
        o[2 * i + h] = *reinterpret_cast<const uint32_t *>(&v);
      }
    }
  }
}

// Writes 4 consecutive output channels of one token row (S > 1 path).
template <int MODE>
// sw, b: the four channels' weight scales and biases; sx: the token's scale
// (staged in shared memory by the caller).
__device__ __forceinline__ void store4(const SwapParams &p, int m, int n, const uint32_t (&v)[4], const float *sw,
                                       const float *b, float sx) {
  if constexpr (MODE == kSwapI8Raw) {
    *reinterpret_cast<uint4 *>((int32_t *)p.y + (size_t)m * p.N + n) = make_uint4(v[0], v[1], v[2], v[3]);
  } else {
    uint32_t o[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float a[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int k = 2 * h + e;
        const float acc = MODE == kSwapW8A16 ? __uint_as_float(v[k]) : (float)(int)v[k];
        a[e] = acc * (sx * sw[k]);
        if (p.bias) a[e] += b[k];
      }
      o[h] = pack_bf16x2(a[0], a[1]);
    }
    *reinterpret_cast<uint2 *>((uint16_t *)p.y + (size_t)m * p.N + n) = make_uint2(o[0], o[1]);
  }
}

// Merged gate_up (S > 1 path): 4 consecutive output channels of one token row
// from the summed gate and up accumulators: y = silu(gate) * up.
// swg, bg4 / swu, bu4: the gate and up channels' weight scales and biases; sx:
// the token's scale (staged in shared memory by the caller; zero biases when
// there is no bias).
template <int MODE>
__device__ __forceinline__ void glu_store4(const SwapParams &p, int m, int ch, const uint32_t (&g)[4],
                                           const uint32_t (&u)[4], const float *swg, const float *bg4,
                                           const float *swu, const float *bu4, float sx) {
  float y[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float ga = MODE == kSwapW8A16 ? __uint_as_float(g[e]) : (float)(int)g[e];
    const float ua = MODE == kSwapW8A16 ? __uint_as_float(u[e]) : (float)(int)u[e];
    const float gv = fmaf(ga, sx * swg[e], bg4[e]);
    const float uv = fmaf(ua, sx * swu[e], bu4[e]);
    y[e] = silu_f(gv) * uv;
  }
  *reinterpret_cast<uint2 *>((uint16_t *)p.y + (size_t)m * p.N + ch) =
      make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
}

template <int BNT, int QT, int MODE>
__global__ void __launch_bounds__(640, 1)
    k_w8_dq(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x, SwapParams p) {
  using C = DqCfg<BNT, MODE>;
  constexpr bool kI8 = MODE != kSwapW8A16;
  constexpr bool kXQ = MODE == kSwapI8Fused;  // quantize the activation tiles in place
  // k-blocks per exactly accumulated chunk: an accumulator takes at most 16 blocks
  // (1024 products of |q| <= 127), so its sum stays an integer below 2^24
  constexpr int CH = kI8 ? 16 : (1 << 30);
  static_assert(!kI8 || BNT <= 64 || C::TSUM, "int32 sums live in registers or in tensor memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *xs = smem + C::X_OFF, *raws = smem + C::RAW_OFF;
  uint64_t *bars = (uint64_t *)(smem + C::BAR_OFF);
  uint64_t *raw_full = bars, *raw_empty = raw_full + C::R;
  uint64_t *x_full = raw_empty + C::R, *x_empty = x_full + C::X;
  uint64_t *a_full = x_empty + C::X, *a_empty = a_full + C::NA;
  uint64_t *acc_full = a_empty + C::NA, *acc_empty = acc_full + C::ND;
  // merged gate_up exchange, per slot: g_ready, u_ready (the writers' two warps arrive),
  // g_taken, u_taken (the readers' two warps arrive)
  uint64_t *g_ready = acc_empty + C::ND, *u_ready = g_ready + 2, *g_taken = u_ready + 2, *u_taken = g_taken + 2;
  uint32_t *tmem_slot = (uint32_t *)(u_taken + 2);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
  float *xchg = reinterpret_cast<float *>(smem + C::XCHG_OFF);
  float *scl_w = reinterpret_cast<float *>(smem + C::SCL_OFF), *scl_b = scl_w + C::BM, *scl_x = scl_b + C::BM;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.z, S = p.splits;
  // The split-K reduction reads the partial tiles of S cluster peers through
  // distributed shared memory: without that cluster shape, report and leave
  // before any barrier, TMEM or peer is touched.
  if (S > 1 && (int)cluster_nctarank() != S) {
    if (threadIdx.x == 0) set_status(p.status, QLIN_ERR_UNSUPPORTED);
    return;
  }
  const int KB = (p.K + C::BK - 1) / C::BK;
  const int kb0 = (int)((int64_t)split * KB / S), kb1 = (int)((int64_t)(split + 1) * KB / S);
  const int nkb = kb1 - kb0;
  const int G = gridDim.x;
  const int my_units = (p.units - (int)blockIdx.x + G - 1) / G;
  const int total = my_units * nkb;
  const int chunks_per_unit = (nkb + CH - 1) / CH;

  {  // barrier initialisation spread over the threads (one barrier each)
    const int t = threadIdx.x;
    constexpr int B0 = C::R, B1 = 2 * C::R, B2 = B1 + C::X, B3 = B2 + C::X, B4 = B3 + C::NA, B5 = B4 + C::NA,
                  B6 = B5 + C::ND, B7 = B6 + C::ND, B8 = B7 + 8;
    static_assert(B8 < C::THREADS, "one thread per barrier");
    uint64_t *bar = nullptr;
    uint32_t cnt = 1;
    if (t < B0) bar = &raw_full[t];
    else if (t < B1) bar = &raw_empty[t - B0], cnt = 4;  // the four warps of the quad that read it
    else if (t < B2) bar = &x_full[t - B1];
    else if (t < B3) bar = &x_empty[t - B2];
    else if (t < B4) bar = &a_full[t - B3], cnt = C::XA ? 5 : 4;  // the converter quad (+ the activation tile)
    else if (t < B5) bar = &a_empty[t - B4];
    else if (t < B6) bar = &acc_full[t - B5], cnt = C::ISSUERS;  // one commit per MMA issuer
    else if (t < B7) bar = &acc_empty[t - B6], cnt = 4;          // the epilogue quad
    else if (t < B8) bar = &g_ready[t - B7], cnt = 2;            // exchange barriers: two warps each
    if (bar) {
      mbar_init(bar, cnt);
      fence_barrier_init();
    }
    if (t == C::THREADS - 1) {
      *abort_flag = 0;
      tma_prefetch_desc(&tm_w);
      tma_prefetch_desc(&tm_x);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Every role but the weight producer waits for the previous kernel of the
  // stream here.  Weight codes are never written by a kernel that lets this one
  // start early (the weight quantizer lets no later kernel start before it
  // completes), so the weight tiles stream from the start.
  if (warp != 0) {
    pdl_wait();
    pdl_trigger();
  }

  if (warp == 0) {  // ------------------------ weight-tile producer
    if (lane == 0) {
      int i = 0;
      for (int j = 0; j < my_units && !*abort_flag; ++j) {
        const int tt = (blockIdx.x + j * G) % p.ntiles;
        for (int kb = 0; kb < nkb; ++kb, ++i) {
          const int s = i % C::R;
          if (i >= C::R && !mbar_wait(&raw_empty[s], ((i / C::R) & 1) ^ 1, abort_flag)) {
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&raw_full[s], C::RAW_BYTES);
          uint8_t *dst = raws + s * C::RAW_BYTES;
          if (p.glu) {  // 64 gate rows, then their 64 up rows (the 64-byte swizzle repeats every 8 rows)
            tma_load_2d(&tm_w, &raw_full[s], dst, (kb0 + kb) * C::BK, tt * 64);
            tma_load_2d(&tm_w, &raw_full[s], dst + 64 * C::BK, (kb0 + kb) * C::BK, p.N + tt * 64);
          } else {
            tma_load_2d(&tm_w, &raw_full[s], dst, (kb0 + kb) * C::BK, tt * C::BM);
          }
        }
      }
      if (*abort_flag) drain_ring(raw_full, C::R, i, C::R);  // abort: armed stages land first
    }
  } else if (warp == 2) {  // ----------------- activation-tile producer
    if (lane == 0) {
      int i = 0;
      for (int j = 0; j < my_units && !*abort_flag; ++j) {
        const int m0 = ((blockIdx.x + j * G) / p.ntiles) * BNT;
        for (int kb = 0; kb < nkb; ++kb, ++i) {
          const int s = i % C::X;
          // the slot is free once the MMA of block i - X is done: XA reads that from
          // the block's A-stage release (one commit per block serves both rings;
          // this thread waits on every block's in turn, and X <= NA keeps it within
          // one phase of each slot)
          if (i >= C::X && !(C::XA ? mbar_wait(&a_empty[(i - C::X) % C::NA], ((i - C::X) / C::NA) & 1, abort_flag)
                                   : mbar_wait(&x_empty[s], ((i / C::X) & 1) ^ 1, abort_flag))) {
            *abort_flag = 1;
            break;
          }
          uint64_t *bar = C::XA ? &a_full[i % C::NA] : &x_full[s];
          mbar_arrive_expect_tx(bar, C::X_BYTES);
          tma_load_2d(&tm_x, bar, xs + s * C::X_BYTES, (kb0 + kb) * C::BK, m0);
        }
      }
      // abort: armed stages land first (XA: the last X blocks' a_full phases, bounded
      // waits that may also run out for want of the quads' arrivals)
      if (*abort_flag) {
        if (C::XA) drain_ring(a_full, C::NA, i, C::X);
        else drain_ring(x_full, C::X, i, C::X);
      }
    }
  } else if (warp == 1 || (warp == 3 && C::ISSUERS == 2)) {  // -- MMA issuers
    // Issuer e (warp 1: e = 0, warp 3: e = 1) takes the k-blocks with kb % ISSUERS == e
    // and accumulates them into its own accumulator tiles (kb % NACC).  The MMA
    // instructions of a block are straight-line code followed by unconditional
    // commits: that keeps one thread issuing an MMA every few dozen cycles.
    if (lane == 0) {
      const int e = warp == 1 ? 0 : 1;
      bool ok = true;
      int cidx = 0;    // chunk counter (same sequence as the epilogue's)
      int last = -1;   // this issuer's last block
      for (int j = 0; j < my_units && ok; ++j) {
        for (int cb = 0; cb < nkb && ok; cb += CH, ++cidx) {  // chunk = k-blocks [cb, ce)
          const int ce = min(nkb, cb + CH);
          const int db = cidx % C::ND;
          if (cidx >= C::ND && !mbar_wait(&acc_empty[db], ((cidx / C::ND) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dset = tmem + db * C::DSTRIDE;
          for (int kb = cb + e; kb < ce; kb += C::ISSUERS) {
            const int i = j * nkb + kb;  // block index within this CTA
            const int sx = i % C::X, sa = i % C::NA;
            if (!mbar_wait(&a_full[sa], (i / C::NA) & 1, abort_flag)) {  // weights and activations
              ok = false;
              break;
            }
            tc_fence_after();
            const int rel = kb - cb;
            const uint32_t dt = dset + (rel % C::NACC) * BNT, at = tmem + C::ACOL + sa * 32;
            const uint32_t acc0 = rel < C::NACC ? 0u : 1u;  // first block of its accumulator starts it
            const uint64_t bd = umma_desc_sw128(smem_u32(xs + sx * C::X_BYTES));
            mma_bf16_ts(dt, at, bd, C::IDESC, acc0);
            mma_bf16_ts(dt, at + 8, bd + 2, C::IDESC, 1u);
            mma_bf16_ts(dt, at + 16, bd + 4, C::IDESC, 1u);
            mma_bf16_ts(dt, at + 24, bd + 6, C::IDESC, 1u);
            if (!C::XA) mma_commit(&x_empty[sx]);
            mma_commit(&a_empty[sa]);
            last = i;
          }
          if (!ok) break;
          mma_commit(&acc_full[db]);  // arrives when this issuer's MMAs of the chunk are done
        }
      }
      // Drain: the CTA must not exit with a commit arrival still in flight towards
      // its shared memory (a successor CTA on this SM may already own it); the
      // waits hold on the abort path too
      if (last >= 0) {
        ok = (C::XA || mbar_wait_drain(&x_empty[last % C::X], (last / C::X) & 1)) &&
             mbar_wait_drain(&a_empty[last % C::NA], (last / C::NA) & 1) && ok;
      }
      if (!ok) *abort_flag = 1;
    }
  } else if (warp >= 4 && warp < 16) {  // ----- converter quads
    const int quad = (warp - 4) >> 2, q4 = warp & 3, row = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    bool ok = true;
    Scale xsc{1.0f, 1.0f, true};
    if constexpr (kXQ) xsc = make_scale(__ldg(p.x_scale));
    for (int i = quad; i < total; i += C::QUADS) {
      const int r = i % C::R, sa = i % C::NA;
      if (!mbar_wait(&raw_full[r], (i / C::R) & 1, abort_flag)) {
        ok = false;
        break;
      }
      // row `row` of the raw tile: four 16-byte chunks, 64-byte swizzle (chunk ^ ((row >> 1) & 3))
      const uint32_t rb = smem_u32(raws + r * C::RAW_BYTES) + row * 64;
      const int sw = (row >> 1) & 3;
      uint4 raw[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) raw[c] = lds128(rb + ((c ^ sw) << 4));
      uint32_t words[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) convert16<QT>(raw[c], words + 8 * c);
      __syncwarp();
      if (lane == 0) mbar_arrive(&raw_empty[r]);
      if constexpr (kXQ) {
        // quantize this block's activation tile in place: thread `row` takes BNT
        // consecutive bytes (BNT / 2 BF16 values) of the BNT x 128-byte tile; the
        // 128-byte swizzle only permutes elements, so the in-place map is the same
        const int sxs = i % C::X;
        if (!mbar_wait(&x_full[sxs], (i / C::X) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t xb = smem_u32(xs + sxs * C::X_BYTES) + row * BNT;
#pragma unroll
        for (int c = 0; c < BNT / 16; ++c) {
          const uint4 v = lds128(xb + 16 * c);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = quantize_i8_value(bf16_bits_to_f32(w[e] & 0xFFFFu), xsc);
            const float hi = quantize_i8_value(bf16_bits_to_f32(w[e] >> 16), xsc);
            o[e] = pack_code_bf16x2(lo, hi);
          }
          sts128(xb + 16 * c, make_uint4(o[0], o[1], o[2], o[3]));
        }
        fence_proxy_async_smem();  // the MMA reads the tile through the async proxy
      }
      if (i >= C::NA && !mbar_wait(&a_empty[sa], ((i / C::NA) & 1) ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      tmem_st32(tmem + lane_base + C::ACOL + sa * 32, words);
      tmem_st_wait();
      // the block's activation tile (already waited for when quantized in place)
      if (C::QX && !kXQ && !mbar_wait(&x_full[i % C::X], (i / C::X) & 1, abort_flag)) {  // XA: on a_full
        ok = false;
        break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[sa]);
    }
    if (!ok) *abort_flag = 1;
  } else if (warp >= 16) {  // ------------------ epilogue quad
    const int q4 = warp & 3, nl = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const bool up_row = p.glu && nl >= 64;  // merged gate_up: TMEM lanes 64..127 hold the up rows
    if (S > 1) {
      // Split-K (one unit per CTA): the factors the cluster's sum applies, read
      // while the main loop runs instead of after the sum.
      const int u = blockIdx.x, tn = u % p.ntiles, mu = (u / p.ntiles) * BNT;
      const int ch = p.glu ? (up_row ? p.N + tn * 64 + (nl - 64) : tn * 64 + nl) : tn * C::BM + nl;
      const bool in = p.glu || ch < p.N;
      // (the raw int32 form has no factors: its scale pointers are null)
      scl_w[nl] = MODE != kSwapI8Raw && in ? __ldg(p.w_scale + ch) : 0.0f;
      scl_b[nl] = MODE != kSwapI8Raw && in && p.bias ? bf16_bits_to_f32(__ldg(p.bias + ch)) : 0.0f;
      for (int t = nl; t < BNT; t += 128)
        scl_x[t] = MODE == kSwapI8Scaled || MODE == kSwapI8Fused
                       ? (p.xs_per_token ? (mu + t < p.M ? __ldg(p.x_scale + mu + t) : 0.0f) : __ldg(p.x_scale))
                       : 1.0f;
    }
    int cidx = 0, xround = 0;
    bool ok = true;
    // Writes the outputs of this thread's row for tokens m0 + c .. m0 + c + 15 from
    // their fp32 values (scale and bias applied).  Merged gate_up: gate row n and
    // up row n are in different warps; the gate rows' threads hand g of tokens
    // 8..15 to the up rows' threads and receive u of tokens 0..7, then each side
    // stores silu(g) * u for its half of the tokens (shared-memory slots with
    // mbarriers, bounded waits).  Returns false if a wait ran out.  All four
    // warps call it equally often.
    auto emit16 = [&](int m0, int c, int ochan, const float (&v)[16]) -> bool {
      uint16_t *y = (uint16_t *)p.y;
      if (!p.glu) {
        // Transpose through this warp's 1 KB of the exchange area (two slots): each
        // thread writes its channel for the 16 tokens, then lane l stores 8
        // consecutive channels of token row (l / 4) and (l / 4) + 8 as one 16-byte
        // vector.  N is a multiple of 16, so a chunk of 8 channels is all in or out.
        uint16_t *stg = reinterpret_cast<uint16_t *>(xchg) + (q4 * 2 + (xround++ & 1)) * 16 * 32;
#pragma unroll
        for (int e = 0; e < 16; ++e) stg[e * 32 + lane] = f32_to_bf16_bits(v[e]);
        __syncwarp();
        const int ch = ochan - lane + (lane & 3) * 8;  // the warp's first channel + this lane's chunk
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = (lane >> 2) + 8 * h, m = m0 + c + r;
          const uint4 vec = *reinterpret_cast<const uint4 *>(stg + r * 32 + (lane & 3) * 8);
          if (m < p.M && ch < p.N) *reinterpret_cast<uint4 *>(y + (size_t)m * p.N + ch) = vec;
        }
        __syncwarp();
        return true;
      }
      const int k = xround++, slot = k & 1, use = k >> 1;  // use: how often this slot was used before
      const int col = nl & 63;
      float *mine = xchg + (slot * 2 + (up_row ? 1 : 0)) * 8 * 64;  // gate: [slot][0], up: [slot][1]
      float *theirs = xchg + (slot * 2 + (up_row ? 0 : 1)) * 8 * 64;
      uint64_t *my_ready = (up_row ? u_ready : g_ready) + slot, *their_ready = (up_row ? g_ready : u_ready) + slot;
      uint64_t *my_taken = (up_row ? u_taken : g_taken) + slot, *their_taken = (up_row ? g_taken : u_taken) + slot;
      // 1. the other side has read what this side wrote into the slot last time
      const bool w0 = use == 0 || mbar_wait(my_taken, (use - 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, w0)) return false;
      // the up rows hand over tokens 0..7 and keep 8..15, the gate rows the other way
      // round (selects between constant indices keep v[] in registers)
      const int keep = up_row ? 8 : 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) mine[e * 64 + col] = up_row ? v[e] : v[8 + e];
      __syncwarp();
      if (lane == 0) mbar_arrive(my_ready);
      // 2. the other side's values for the tokens this side stores
      const bool w1 = mbar_wait(their_ready, use & 1, abort_flag);
      if (!__all_sync(0xffffffffu, w1)) return false;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float other = theirs[e * 64 + col];
        const float own = up_row ? v[8 + e] : v[e];
        const float g = up_row ? other : own, u = up_row ? own : other;
        const int m = m0 + c + keep + e;
        if (m < p.M) y[(size_t)m * p.N + ochan] = f32_to_bf16_bits(silu_f(g) * u);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(their_taken);
      return true;
    };
    for (int j = 0; j < my_units && ok; ++j) {
      const int u = blockIdx.x + j * G;
      const int tt = u % p.ntiles, m0 = (u / p.ntiles) * BNT;
      // weight row of this TMEM lane and the output channel it writes
      const int wrow = !p.glu ? tt * C::BM + nl : (up_row ? p.N + tt * 64 + (nl - 64) : tt * 64 + nl);
      const int ochan = p.glu ? tt * 64 + (nl & 63) : wrow;
      const bool valid = p.glu ? true : wrow < p.N;
      // this row's factors (used without split-K), read before the accumulator
      // wait where the registers allow (not beside 64 int32 sums)
      constexpr bool kEarly = !(kI8 && !C::TSUM && BNT >= 64);
      // (the raw int32 form has no factors: its scale pointers are null)
      auto row_factors = [&](float &sw, float &b, float &sx) {
        constexpr bool kScaled = MODE != kSwapI8Raw;
        sw = kScaled && S == 1 && valid ? __ldg(p.w_scale + wrow) : 0.0f;
        b = kScaled && S == 1 && valid && p.bias ? bf16_bits_to_f32(__ldg(p.bias + wrow)) : 0.0f;
        sx = kScaled && kI8 && S == 1 ? __ldg(p.x_scale) : 1.0f;
      };
      float sw_u = 0.0f, b_u = 0.0f, sx_u = 1.0f;
      if constexpr (kEarly) row_factors(sw_u, b_u, sx_u);
      constexpr int NSUM = kI8 && !C::TSUM ? BNT : 1;  // int32 sums held in registers
      int32_t sums[NSUM];
#pragma unroll
      for (int c = 0; c < NSUM; ++c) sums[c] = 0;
      for (int ch = 0; ch < chunks_per_unit && ok; ++ch, ++cidx) {
        const int db = cidx % C::ND;
        ok = mbar_wait(&acc_full[db], (cidx / C::ND) & 1, abort_flag);
        tc_fence_after();
        // tcgen05.ld is warp-collective: every lane of the warp takes the same path
        const bool run = __all_sync(0xffffffffu, ok && !*abort_flag);
        if (!run) {
          ok = false;
          break;
        }
        const uint32_t dt = tmem + lane_base + db * C::DSTRIDE;
        const int in_chunk = min(CH, nkb - ch * CH);
        const int nacc = in_chunk < C::NACC ? in_chunk : C::NACC;  // accumulators written in this chunk
        // 16 columns of the chunk's sum: accumulators added in a fixed order (all
        // of a chunk's tensor-memory loads are issued before the one wait)
        auto load16 = [&](int c, uint32_t (&r)[16]) {
          if constexpr (C::NACC == 1) {
            tmem_ld16(dt + c, r);
            tmem_ld_wait();
          } else if constexpr (C::NACC > 2) {
            // four small accumulators (16/32-token tiles, a short epilogue): one at a time
            tmem_ld16(dt + c, r);
            tmem_ld_wait();
            for (int a = 1; a < nacc; ++a) {
              uint32_t t[16];
              tmem_ld16(dt + a * BNT + c, t);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(t[e]));
            }
          } else {
            // two accumulators: both loads in flight per wait
            uint32_t t[16];
            tmem_ld16(dt + c, r);
            if (nacc > 1) tmem_ld16(dt + BNT + c, t);
            tmem_ld_wait();
            if (nacc > 1) {
#pragma unroll
              for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(t[e]));
            }
#pragma unroll
            for (int a = 2; a < C::NACC; a += 2) {
              if (a < nacc) {
                uint32_t u[16];
                tmem_ld16(dt + a * BNT + c, t);
                if (a + 1 < nacc) tmem_ld16(dt + (a + 1) * BNT + c, u);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(t[e]));
                if (a + 1 < nacc) {
#pragma unroll
                  for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(u[e]));
                }
              }
            }
          }
        };
        if constexpr (kI8 && C::TSUM) {
          // the accumulator holds exact integers below 2^23: fold them into the int32
          // running sums in tensor memory (the first chunk of a tile starts them)
          const uint32_t ts = tmem + lane_base + C::SUMCOL;
#pragma unroll 1
          for (int c = 0; c < BNT; c += 16) {
            uint32_t r[16], u[16];
            tmem_ld16(dt + c, r);
            if (ch > 0) tmem_ld16(ts + c, u);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e)
              u[e] = (uint32_t)((ch > 0 ? (int32_t)u[e] : 0) + __float2int_rn(__uint_as_float(r[e])));
            tmem_st16(ts + c, u);
          }
          tmem_st_wait();
        } else if constexpr (kI8) {
          // each accumulator holds an exact integer below 2^23: convert, then add in int32
          for (int a = 0; a < nacc; ++a) {
#pragma unroll
            for (int c = 0; c < BNT; c += 16) {
              uint32_t r[16];
              tmem_ld16(dt + a * BNT + c, r);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) sums[c + e] += __float2int_rn(__uint_as_float(r[e]));
            }
          }
        } else if (S == 1) {
          if constexpr (!kEarly) row_factors(sw_u, b_u, sx_u);
          const float sw = sw_u, b = b_u;
          if constexpr (C::NACC == 1) {
            // double-buffered: the next 16 columns are loaded while these are stored
            uint32_t ra[16], rb[16];
            tmem_ld16(dt, ra);
#pragma unroll 1
            for (int c = 0; c < BNT && ok; c += 32) {
              tmem_ld_wait();
              if (c + 16 < BNT) tmem_ld16(dt + c + 16, rb);
              float v[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = fmaf(__uint_as_float(ra[e]), sw, b);
              ok = emit16(m0, c, ochan, v);
              if (c + 16 >= BNT) break;
              tmem_ld_wait();
              if (c + 32 < BNT) tmem_ld16(dt + c + 32, ra);
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = fmaf(__uint_as_float(rb[e]), sw, b);
              ok = ok && emit16(m0, c + 16, ochan, v);
            }
            tmem_ld_wait();  // no load left in flight past the accumulator release
          } else {
#pragma unroll 1
            for (int c = 0; c < BNT && ok; c += 16) {
              uint32_t r[16];
              load16(c, r);
              float v[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = fmaf(__uint_as_float(r[e]), sw, b);
              ok = emit16(m0, c, ochan, v);
            }
          }
        } else {
          uint32_t *red = reinterpret_cast<uint32_t *>(smem);  // partial tile, [token][channel]
#pragma unroll 1
          for (int c = 0; c < BNT; c += 16) {
            uint32_t r[16];
            load16(c, r);
#pragma unroll
            for (int e = 0; e < 16; ++e) red[(c + e) * C::BM + nl] = r[e];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[db]);
      }
      if constexpr (kI8) {
        // the tile's int32 sums of tokens c..c+15: from registers, or from tensor memory
        auto sums16 = [&](int c, int32_t (&s16)[16]) {
          if constexpr (C::TSUM) {
            uint32_t u[16];
            tmem_ld16(tmem + lane_base + C::SUMCOL + c, u);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) s16[e] = (int32_t)u[e];
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) s16[e] = sums[(c + e) % NSUM];
          }
        };
        if (ok) {
          if (S == 1) {
            if constexpr (MODE == kSwapI8Raw) {
#pragma unroll
              for (int c = 0; c < BNT; c += 16) {  // fully unrolled: sums[] stays in registers
                int32_t s16[16];
                sums16(c, s16);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  if (valid && m0 + c + e < p.M) ((int32_t *)p.y)[(size_t)(m0 + c + e) * p.N + wrow] = s16[e];
              }
            } else {
              if constexpr (!kEarly) row_factors(sw_u, b_u, sx_u);
              const float sw = sw_u, sx0 = sx_u, b = b_u;
#pragma unroll
              for (int c = 0; c < BNT; c += 16) {  // fully unrolled: sums[] stays in registers
                if (ok) {
                  int32_t s16[16];
                  sums16(c, s16);
                  float v[16];
#pragma unroll
                  for (int e = 0; e < 16; ++e) {
                    const int m = m0 + c + e;
                    const float sx = p.xs_per_token ? (m < p.M ? __ldg(p.x_scale + m) : 0.0f) : sx0;
                    v[e] = fmaf((float)s16[e], sx * sw, b);
                  }
                  ok = emit16(m0, c, ochan, v);
                }
              }
            }
          } else {
            int32_t *red = reinterpret_cast<int32_t *>(smem);
#pragma unroll
            for (int c = 0; c < BNT; c += 16) {
              int32_t s16[16];
              sums16(c, s16);
#pragma unroll
              for (int e = 0; e < 16; ++e) red[(c + e) * C::BM + nl] = s16[e];
            }
          }
        }
      }
    }
    if (!ok) *abort_flag = 1;
  }
  if (threadIdx.x == 0 && *abort_flag) set_status(p.status, QLIN_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (S > 1) {  // one unit per CTA: sum the partial tiles of the cluster
    cluster_sync();
    if (warp >= 4 && p.glu) {
      // merged gate_up: a unit is 4 gate rows of one token plus the same 4 up rows (64 rows on)
      const int ct = threadIdx.x - 128;  // 512 threads
      const uint32_t base = smem_u32(smem);
      const int u = blockIdx.x, tt = u % p.ntiles, m0 = (u / p.ntiles) * BNT;
      constexpr int UG = BNT * 64 / 4;
      const int u0 = (int)((int64_t)split * UG / S), u1 = (int)((int64_t)(split + 1) * UG / S);
      for (int g4 = u0 + ct; g4 < u1; g4 += 512) {
        const int jj = g4 / 16, nq = (g4 % 16) * 4;
        const uint32_t wg = (uint32_t)(jj * C::BM + nq), wu = wg + 64;  // word offsets in the tile
        uint32_t ag[4] = {0, 0, 0, 0}, au[4] = {0, 0, 0, 0};
        // RB peers' gate and up pieces in flight at once (one with int32 sums in
        // registers: measured no faster with two, and it leaves them fewer registers)
        constexpr int RB = kI8 && !C::TSUM ? 1 : 2;
        for (int r0 = 0; r0 < S; r0 += RB) {
          uint4 vg[RB], vu[RB];
#pragma unroll
          for (int q = 0; q < RB; ++q)
            if (r0 + q < S) {
              vg[q] = ld_dsmem_v4(map_peer_smem(base + 4u * wg, (uint32_t)(r0 + q)));
              vu[q] = ld_dsmem_v4(map_peer_smem(base + 4u * wu, (uint32_t)(r0 + q)));
            }
#pragma unroll
          for (int q = 0; q < RB; ++q) {  // summed in rank order: deterministic
            if (r0 + q >= S) break;
            const uint32_t g4v[4] = {vg[q].x, vg[q].y, vg[q].z, vg[q].w}, u4v[4] = {vu[q].x, vu[q].y, vu[q].z, vu[q].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              ag[e] = kI8 ? (uint32_t)((int32_t)ag[e] + (int32_t)g4v[e])
                          : __float_as_uint(__uint_as_float(ag[e]) + __uint_as_float(g4v[e]));
              au[e] = kI8 ? (uint32_t)((int32_t)au[e] + (int32_t)u4v[e])
                          : __float_as_uint(__uint_as_float(au[e]) + __uint_as_float(u4v[e]));
            }
          }
        }
        const int m = m0 + jj;
        if (m < p.M)
          glu_store4<MODE>(p, m, tt * 64 + nq, ag, au, scl_w + nq, scl_b + nq, scl_w + 64 + nq, scl_b + 64 + nq,
                           scl_x[jj]);
      }
    } else if (warp >= 4) {
      const int ct = threadIdx.x - 128;  // 512 threads
      const uint32_t base = smem_u32(smem);
      const int u = blockIdx.x, n0 = (u % p.ntiles) * C::BM, m0 = (u / p.ntiles) * BNT;
      constexpr int U = BNT * C::BM / 4;  // 4-word units of the tile
      const int u0 = (int)((int64_t)split * U / S), u1 = (int)((int64_t)(split + 1) * U / S);
      for (int w4 = u0 + ct; w4 < u1; w4 += 512) {
        uint32_t acc[4] = {0, 0, 0, 0};
        // RB peers' pieces in flight at once (one with int32 sums in registers:
        // measured no faster with two, and it leaves them fewer registers)
        constexpr int RB = kI8 && !C::TSUM ? 1 : 4;
        for (int r0 = 0; r0 < S; r0 += RB) {
          uint4 v[RB];
#pragma unroll
          for (int q = 0; q < RB; ++q)
            if (r0 + q < S) v[q] = ld_dsmem_v4(map_peer_smem(base + 16u * w4, (uint32_t)(r0 + q)));
#pragma unroll
          for (int q = 0; q < RB; ++q) {  // summed in rank order: deterministic
            if (r0 + q >= S) break;
            const uint32_t vv[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              acc[e] = kI8 ? (uint32_t)((int32_t)acc[e] + (int32_t)vv[e])
                           : __float_as_uint(__uint_as_float(acc[e]) + __uint_as_float(vv[e]));
          }
        }
        const int e0 = 4 * w4, jj = e0 / C::BM, nl = e0 % C::BM;
        const int m = m0 + jj, n = n0 + nl;
        if (m < p.M && n < p.N) store4<MODE>(p, m, n, acc, scl_w + nl, scl_b + nl, scl_x[jj]);
      }
    }
    cluster_sync();  // no CTA leaves while a peer may still read its shared memory
  }
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ================================================================ launchers
template <class KernelT>
static cudaError_t set_smem(KernelT kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_fp8_gemm(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st) {
  if (g.M == 0) return cudaSuccess;
  using C = Fp8Cfg;
  CUtensorMap ta, tb, ty;
  // glu: the weight has 2N rows and a tile takes 128 gate rows plus their 128 up rows (two boxes)
  const int64_t wrows = g.glu ? 2 * g.N : g.N;
  // B is loaded as two boxes of 128 rows (two halves of the 256-row tile); y [M, N]
  // (N = I for glu) is written in 32 x 32 blocks through a 64-byte-swizzled staging block
  if (!make_map(&ta, g.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.M, g.K, C::BK, C::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&tb, g.qw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, wrows, g.K, C::BK, C::BN / 2,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&ty, g.y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.M, g.N, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  // glu: an output tile is 128 channels (n0 counts the 256 gate+up columns of the MMA tile)
  const int mtiles = (int)((g.M + C::BM - 1) / C::BM);
  const int ntiles = g.glu ? (int)(g.N / (C::BN / 2)) : (int)((g.N + C::BN - 1) / C::BN);
  const int nkb = (int)((g.K + C::BK - 1) / C::BK);
  Fp8Params p{(int)g.M, (int)g.N, (int)g.K, mtiles, ntiles, g.x_scale_per_token, g.glu,
              (uint8_t *)g.a, g.xq_flags, (nkb + 3) / 4 * 4, 1, g.w_scale, g.x_scale,
              g.bias, (uint16_t *)g.y, dev.status};
  if (g.xq) {  // fused quantization: cooperative launch (every CTA resident)
    if (g.x_scale_per_token || !g.xq_flags) return cudaErrorInvalidValue;
    CUtensorMap tx;  // the BF16 activations, chunks of XQ_ROWS rows of a 128 x 128 task tile
    if (!make_map(&tx, g.xq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.M, g.K, C::BK, Fp8CfgT<1, 1>::XQ_ROWS,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    const size_t fb = fp8_xq_flag_bytes(g.M, g.K);
    cudaError_t e = cudaMemsetAsync(g.xq_flags, 0, fb, st);
    if (e != cudaSuccess) return e;
    // CTA pairs (256 x 256 tiles with pair MMAs); cooperative launch of 2-CTA clusters
    using CX = Fp8CfgT<1, 1>;
    static cudaError_t a1 = set_smem(k_fp8_gemm<1, 1>, CX::SMEM);
    if (a1 != cudaSuccess) return a1;
    const int items = ((mtiles + 1) / 2) * ntiles, pairs = dev.sms / 2;
    const int grid = 2 * (items < pairs ? items : pairs);
    // band of quantization tasks: the m-tiles one wave of grid / 2 pair tiles spans
    const int b = 2 * ((grid / 2 + ntiles - 1) / ntiles);
    p.xq_band = b < mtiles ? b : mtiles;
    return launch_kernel_coop(k_fp8_gemm<1, 1>, dim3((unsigned)grid), dim3(CX::THREADS), CX::SMEM, st, 2, ta, tb, tx,
                              ty, p);
  }
  if (mtiles >= 2) {  // CTA pairs: 256 x 256 tiles with pair MMAs
    using CP = Fp8CfgT<0, 1>;
    static cudaError_t attr2 = set_smem(k_fp8_gemm<0, 1>, CP::SMEM);
    if (attr2 != cudaSuccess) return attr2;
    const int items = ((mtiles + 1) / 2) * ntiles, pairs = dev.sms / 2;
    const int grid = 2 * (items < pairs ? items : pairs);
    return launch_kernel_x(k_fp8_gemm<0, 1>, dim3((unsigned)grid), dim3(CP::THREADS), CP::SMEM, st, 2, ta, tb, tb, ty,
                           p);
  }
  static cudaError_t attr = set_smem(k_fp8_gemm<0, 0>, C::SMEM);
  if (attr != cudaSuccess) return attr;
  const int tiles = mtiles * ntiles, grid = tiles < dev.sms ? tiles : dev.sms;
  return launch_kernel(k_fp8_gemm<0, 0>, dim3((unsigned)grid), dim3(C::THREADS), C::SMEM, st, 1, ta, tb, tb, ty, p);
}

// Token tile (MMA N) of the W8A16 swap-AB kernel.  Up to 128 tokens the tile
// covers the batch.  Above that both 128 and 256 are candidates: a 256-token
// tile converts each weight tile once for twice the tokens, a 128-token tile
// makes twice the output tiles (fewer or no K splits, finer waves).  The cost
// of each is estimated as waves x k-blocks per CTA x per-block cost, where a
// 256-token block costs 1.63 times a 128-token block (the ratio of their
// per-unit times measured on the 7B gate_up shape, K = 3584, N = 37888).
// Task flags of the fused-quantization FP8 GEMM: one u32 per (m-tile, 128-k
// block), each m-tile's row padded to a multiple of four (read four at a time),
// then one u32 per band of m-tiles (at most one band per m-tile).
size_t fp8_xq_flag_bytes(int64_t M, int64_t K) {
  const int64_t mtiles = (M + Fp8Cfg::BM - 1) / Fp8Cfg::BM, nkb = (K + Fp8Cfg::BK - 1) / Fp8Cfg::BK;
  return (size_t)(mtiles * ((nkb + 3) / 4 * 4 + 1) * 4);
}

// The fused kernel hides the quantization behind the GEMM's main loop, but its
// shared memory holds the activation ring instead of the staging that lets the
// separate GEMM store its outputs through TMA.  Measured, it wins where each
// tile's main loop is long and the quantization a large share of the work:
// K >= 4096, at most 4096 GEMM columns, and 64 m-tiles or more (8192 tokens);
// at K = 2048 the separate pass with the TMA-store epilogue is 20-28% faster.
// Its quantizers are the GEMM's CTAs, so the pair tiles must fill every SM.
// N counts GEMM columns (2I for the merged gate_up).
// QLIN_FP8_FUSED_QUANT=0 in the environment (read once) keeps the separate
// quantization pass everywhere, so the two forms can be compared on one shape.
bool fp8_xq_used(int64_t M, int64_t K, int64_t N, int sms) {
  static const bool enabled = [] {
    const char *v = std::getenv("QLIN_FP8_FUSED_QUANT");
    return !(v && v[0] == '0' && v[1] == 0);
  }();
  if (!enabled) return false;
  const int64_t mtiles = (M + Fp8Cfg::BM - 1) / Fp8Cfg::BM, ntiles = (N + Fp8Cfg::BN - 1) / Fp8Cfg::BN;
  return mtiles >= 64 && K >= 4096 && N <= 4096 && ((mtiles + 1) / 2) * ntiles >= sms / 2;
}

int w8_swap_bnt(int64_t M, int64_t N, int64_t K, int sms) {
  if (M <= 128) return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
  const int64_t kb = (K + 63) / 64, nt = (N + 127) / 128;
  auto cost = [&](int bnt, double per_block) {
    const int64_t units = nt * ((M + bnt - 1) / bnt);
    const int64_t s = w8_swap_splits(units, K, sms, bnt);
    const int64_t waves = (units * s + sms - 1) / sms;
    return (double)waves * (double)((kb + s - 1) / s) * per_block;
  };
  return cost(128, 1.0) < cost(256, 1.63) ? 128 : 256;
}
int i8_swap_bnt(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

// Split-K factor: CTAs of a cluster that share one output tile when the tiles
// alone cannot fill the GPU.  Each CTA of a cluster stages a 128 x BNT fp32
// partial tile and reduces 1/S of the tile over all S peers, so for token tiles
// of 128 or more the split is capped at 4 and keeps at least 8 k-blocks a CTA
// (measured: q/down projections at 256 tokens took twice as long with 8 splits).
int w8_swap_splits(int64_t tiles, int64_t K, int sms, int bnt) {
  const int64_t kb = (K + 63) / 64;
  if (tiles * 4 >= (int64_t)sms * 3) return 1;
  int64_t s = sms / tiles;
  const int64_t cap = bnt >= 128 ? 4 : 8, min_blocks = bnt >= 128 ? 8 : 2;
  if (s > cap) s = cap;
  if (s > kb / min_blocks) s = kb / min_blocks;
  return s < 1 ? 1 : (int)s;
}

template <int BNT, int QT, int MODE>
static cudaError_t launch_dq_t(const GemmArgs &g, const void *xb, const DeviceInfo &dev, cudaStream_t st) {
  using C = DqCfg<BNT, MODE>;
  CUtensorMap tw, tx;
  // glu: the weight has 2N rows; a tile loads 64 gate rows and their 64 up rows (two boxes)
  const int64_t wrows = g.glu ? 2 * g.N : g.N;
  if (!make_map(&tw, g.qw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, wrows, g.K, C::BK, g.glu ? 64 : C::BM,
                CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&tx, xb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.M, g.K, C::BK, BNT, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static cudaError_t attr = set_smem(k_w8_dq<BNT, QT, MODE>, C::SMEM);
  if (attr != cudaSuccess) return attr;
  const int ntiles = g.glu ? (int)(g.N / 64) : (int)((g.N + C::BM - 1) / C::BM);
  const int units = ntiles * (int)((g.M + BNT - 1) / BNT);
  int S = w8_swap_splits(units, g.K, dev.sms, BNT);
  // A unit's splits reduce through their cluster, and every unit's cluster
  // should be resident in one wave: fewer splits where the GPCs cannot hold
  // `units` clusters of S CTAs at once (a second wave doubles the call).
  static std::atomic<int> clusters[kMaxDevices * 9];
  for (int mc; S > 1 && (mc = max_active_clusters_z(k_w8_dq<BNT, QT, MODE>, dim3(C::THREADS), C::SMEM, (unsigned)S,
                                                     dev.device, clusters)) > 0 && units > mc;)
    --S;
  const int G = S > 1 ? units : (units < dev.sms ? units : dev.sms);
  SwapParams p{(int)g.M, (int)g.N, (int)g.K, g.x_scale_per_token, g.glu, S,  units,
               ntiles,    g.w_scale, g.x_scale, g.bias,  g.y,        dev.status};
  return launch_kernel(k_w8_dq<BNT, QT, MODE>, dim3((unsigned)G, 1, (unsigned)S), dim3(C::THREADS), C::SMEM, st,
                       (unsigned)S, tw, tx, p);
}

template <int QT>
static cudaError_t launch_w8a16_q(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st) {
  switch (w8_swap_bnt(g.M, g.glu ? 2 * g.N : g.N, g.K, dev.sms)) {
    case 16: return launch_dq_t<16, QT, kSwapW8A16>(g, g.a, dev, st);
    case 32: return launch_dq_t<32, QT, kSwapW8A16>(g, g.a, dev, st);
    case 64: return launch_dq_t<64, QT, kSwapW8A16>(g, g.a, dev, st);
    case 128: return launch_dq_t<128, QT, kSwapW8A16>(g, g.a, dev, st);
    default: return launch_dq_t<256, QT, kSwapW8A16>(g, g.a, dev, st);
  }
}

cudaError_t launch_w8a16_swap(const GemmArgs &g, const DeviceInfo &dev, cudaStream_t st) {
  if (g.M == 0) return cudaSuccess;
  return g.qtype == QLIN_INT8 ? launch_w8a16_q<QLIN_INT8>(g, dev, st) : launch_w8a16_q<QLIN_E4M3>(g, dev, st);
}

// INT8 x INT8 on the BF16 tensor cores; `xb` holds the activation codes as
// integer-valued BF16 [M, K].  raw: int32 accumulator out; else scaled BF16.
// fused: `xb` is the BF16 activation itself, quantized inside the kernel with
// the static scale (one token tile, M <= 64).
cudaError_t launch_i8_swap(const GemmArgs &g, const void *xb, bool raw, const DeviceInfo &dev, cudaStream_t st,
                           bool fused) {
  if (g.M == 0) return cudaSuccess;
  if (fused) {
    if (raw || g.x_scale_per_token || g.M > 64) return cudaErrorInvalidValue;
    switch (i8_swap_bnt(g.M)) {
      case 16: return launch_dq_t<16, QLIN_INT8, kSwapI8Fused>(g, xb, dev, st);
      case 32: return launch_dq_t<32, QLIN_INT8, kSwapI8Fused>(g, xb, dev, st);
      default: return launch_dq_t<64, QLIN_INT8, kSwapI8Fused>(g, xb, dev, st);
    }
  }
  switch (i8_swap_bnt(g.M)) {
    case 16:
      return raw ? launch_dq_t<16, QLIN_INT8, kSwapI8Raw>(g, xb, dev, st)
                 : launch_dq_t<16, QLIN_INT8, kSwapI8Scaled>(g, xb, dev, st);
    case 32:
      return raw ? launch_dq_t<32, QLIN_INT8, kSwapI8Raw>(g, xb, dev, st)
                 : launch_dq_t<32, QLIN_INT8, kSwapI8Scaled>(g, xb, dev, st);
    case 64:
      return raw ? launch_dq_t<64, QLIN_INT8, kSwapI8Raw>(g, xb, dev, st)
                 : launch_dq_t<64, QLIN_INT8, kSwapI8Scaled>(g, xb, dev, st);
    default:
      return raw ? launch_dq_t<128, QLIN_INT8, kSwapI8Raw>(g, xb, dev, st)
                 : launch_dq_t<128, QLIN_INT8, kSwapI8Scaled>(g, xb, dev, st);
  }
}

}  // namespace qlin
