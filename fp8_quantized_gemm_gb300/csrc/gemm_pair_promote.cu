// Per-K-group GEMM with FP32 scales (Transformers fine-grained FP8, 一:
// C[m, n] = sum over 128-wide K groups g of sa[m, g] * sb[n / 128, g] *
// sum_{k in g} qa[m, k] qb[n, k]) on CTA pairs (tcgen05 cta_group::2).
//
// FP32 scales are not powers of two, so the tensor core cannot apply them:
// every 128-deep K slice is contracted into its own TMEM buffer and the
// epilogue warps promote it, acc += sa * sb * partial, in registers.  Two
// CTAs on neighbouring SMs compute one 256 x 256 tile with M = 256 MMAs
// issued by the even CTA (the leader):
//
//   - each CTA stages its own 128 rows of A and its own 128 rows of B per k
//     block (32 KB a stage, six stages), both CTAs' copies completing on the
//     leader's full barrier;
//   - the leader's MMAs read both CTAs' shared memory at the same offsets
//     and write each CTA's 128 rows of the slice's partial product into that
//     CTA's TMEM, one of two 256-column buffers;
//   - tcgen05.commit multicasts each stage release and each "slice ready" to
//     both CTAs; eight epilogue warps per CTA (two per TMEM lane quadrant,
//     128 columns each) read the slice out in 16-column chunks, each read in
//     flight under the previous chunk's FMAs, and hand the buffer back on
//     the leader's barrier after the last read, so the tensor core runs the
//     next slice meanwhile.
//
// The TMEM reads bound the kernel (the numbers are at the configuration
// below).  A warp's 128 accumulators stay in registers for the whole tile;
// its columns lie in one 128-row block of B, so one weight scale per slice.
// The scales of the next slice are loaded one slice ahead, and their lines
// four slices ahead are brought into L2.
#include "common.cuh"
#include "expert_tiles.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace fp8k {

// 256-row tiles per band of the grouped tile order.
constexpr int64_t kPromoteBandRows = 8;

template <int BN_, int STAGES, int EPI>
struct PromoteCfg {
  // per CTA: 128 rows x BN columns; pair: 256 x BN
  static constexpr int BM = 128, BN = BN_, BK = 128;
  // EPI epilogue warps, EPI / 4 per TMEM lane quadrant, each promoting
  // kCols columns of its 32 rows
  static constexpr int kEpiWarps = EPI;
  static constexpr int kCols = 4 * BN / EPI;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr uint32_t kABytes = BM * BK;
  static constexpr uint32_t kBBytes = (BN / 2) * BK;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTileBytes = STAGES * kStageBytes;
  static constexpr int kAccBufs = 512 / BN;  // 4 x 128, 2 x 192 or 2 x 256 columns
  // the allocation: a power of two columns
  static constexpr uint32_t kTmemCols = kAccBufs * BN <= 256 ? 256u : 512u;
  static constexpr int kNumBars = 2 * STAGES + 2 * kAccBufs + 1;
  static constexpr uint32_t kSmem = 1024 + kTileBytes + 8 * kNumBars + 16;
  static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
  static_assert(kTmemCols <= 512, "TMEM budget");
  static_assert(kSmem <= 227 * 1024, "shared-memory budget");
  static_assert(EPI % 4 == 0 && kCols % 32 == 0, "whole 32-column chunks per warp");
  // a warp's columns start at a multiple of kCols (BN is one), and kCols
  // divides 128: they lie in one 128-row block of B, so one weight scale
  // per warp and slice
  static_assert(128 % kCols == 0 && BN % kCols == 0, "one 128-column B block of scales per warp");
};

template <int BN, int STAGES, int EPI, bool EXPERTS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PromoteCfg<BN, STAGES, EPI>::kThreads, 1)
    gemm_pair_promote_kernel(const __grid_constant__ CUtensorMap tma,
                             const __grid_constant__ CUtensorMap tmb, const GemmArgs args) {
  using C = PromoteCfg<BN, STAGES, EPI>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kTileBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const DevErr err{args.err, args.wait_limit_ns};

  auto sA = [&](int s) { return smem_u32(smem + s * C::kStageBytes); };
  auto sB = [&](int s) { return smem_u32(smem + s * C::kStageBytes + C::kABytes); };
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
  auto accf_bar = [&](int b) { return smem_u32(&bars[2 * STAGES + b]); };
  auto acce_bar = [&](int b) { return smem_u32(&bars[2 * STAGES + C::kAccBufs + b]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * STAGES + 2 * C::kAccBufs]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 2 * C::kEpiWarps);  // both CTAs' epilogue warps
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma);
    tma_prefetch_desc(&tmb);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);

  const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int64_t rows = (args.M + 255) / 256, tiles_n = (args.N + C::BN - 1) / C::BN;
  // Expert-grouped rows (MoE): a tile never spans two experts; expert e
  // owns ceil(rows_e / 256) * tiles_n consecutive tile indices
  // (expert_tiles.cuh).  Both CTAs of a pair read the same offsets, so they
  // agree on every tile.
  __shared__ ExpertTiles<EXPERTS> ex;
  const int E = EXPERTS ? args.experts : 0;
  if constexpr (EXPERTS) {
    if (warp == 0) build_expert_tiles(args.offsets, E, args.M, tiles_n, 256, lane, ex);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barrier inits visible to the peer before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t num_tiles = EXPERTS ? ex.tile0[E] : rows * tiles_n;
  const int kb_count = (int)(args.K / C::BK);
  // Tile t: rows [m0, row_end) of A and C (row_end ends the expert's rows),
  // columns [n0, n0 + BN), B tensor-map row brow, scale offset sbo.  Pair p
  // takes tiles p, p + npairs, ...; plain rows go in the grouped order
  // (bands of kPromoteBandRows 256-row tiles walked column by column, so
  // the pairs in flight share A and B blocks in L2), expert rows expert by
  // expert, row tile by row tile.
  struct TileInfo {
    int64_t m0, n0, row_end, brow, sbo;
  };
  auto tile_info = [&](int64_t t) {
    TileInfo ti;
    if constexpr (EXPERTS) {
      const int lo = expert_of_tile(ex, E, t);
      const int64_t local = t - ex.tile0[lo];
      ti.m0 = ex.row0[lo] + (local / tiles_n) * 256;
      ti.n0 = (local % tiles_n) * C::BN;
      ti.row_end = ex.row0[lo + 1];
      ti.brow = (int64_t)lo * args.N + ti.n0;
      ti.sbo = (int64_t)lo * args.sb_expert_stride;
    } else {
      // (32-bit: tile counts fit, and the 64-bit division's register needs
      // would meet the accumulators)
      const uint32_t tn = (uint32_t)tiles_n, t32 = (uint32_t)t;
      const uint32_t band = t32 / ((uint32_t)kPromoteBandRows * tn);
      const uint32_t left = (uint32_t)rows - band * (uint32_t)kPromoteBandRows;
      const uint32_t band_rows = left < (uint32_t)kPromoteBandRows ? left : (uint32_t)kPromoteBandRows;
      const uint32_t local = t32 - band * (uint32_t)kPromoteBandRows * tn;
      ti.m0 = (int64_t)(band * (uint32_t)kPromoteBandRows + local % band_rows) * 256;
      ti.n0 = (int64_t)(local / band_rows) * C::BN;
      ti.row_end = args.M;
      ti.brow = ti.n0;
      ti.sbo = 0;
    }
    return ti;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint32_t full_leader0 = mapa_shared(full_bar(0), 0);
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = pair; t < num_tiles && ok; t += npairs) {
      const TileInfo ti = tile_info(t);
      const int32_t am = (int32_t)(ti.m0 + rank * C::BM);
      const int32_t bn = (int32_t)(ti.brow + rank * (C::BN / 2));
      for (int kb = 0; kb < kb_count; ++kb, ++it) {
        const int s = (int)(it % STAGES);
        const uint32_t round = it / STAGES;
        if (!mbar_wait_warp(empty_bar(s), (round & 1u) ^ 1u, abort_flag, err, 1)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          const int32_t k0 = kb * C::BK;
          if (leader) {
            mbar_arrive_expect_tx(full_bar(s), 2 * C::kStageBytes);
            tma_load_2d(sA(s), &tma, full_bar(s), k0, am);
            tma_load_2d(sB(s), &tmb, full_bar(s), k0, bn);
          } else {
            const uint32_t fb = full_leader0 + 8u * (uint32_t)s;
            tma_load_2d_pair(sA(s), &tma, fb, k0, am);
            tma_load_2d_pair(sB(s), &tmb, fb, k0, bn);
          }
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      if (leader) {
        const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
        for (uint32_t i = first; i < it; ++i) drain_wait(full_bar(i % STAGES), (i / STAGES) & 1u);
      } else {
        drain_wait(drain_bar, 0);  // nothing arrives here: a fixed 20 ms grace period
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------- MMA (leader only)
    if (leader && elect_one()) {
      const uint32_t idesc = idesc_f8f6f4(256, C::BN, args.fa, args.fb);
      uint32_t it = 0;
      bool ok = true;
      for (int64_t t = pair; t < num_tiles && ok; t += npairs) {
        for (int kb = 0; kb < kb_count; ++kb, ++it) {
          // one k block per accumulator use: stage it % STAGES, buffer it % 4
          const int s = (int)(it % STAGES);
          const uint32_t buf = it % C::kAccBufs, use = it / C::kAccBufs;
          if (!mbar_wait(acce_bar(buf), (use & 1u) ^ 1u, abort_flag, err, 2) ||
              !mbar_wait(full_bar(s), (it / STAGES) & 1u, abort_flag, err, 2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const OperandDesc ad = operand_desc(sA(s), 0, C::kABytes);
          const OperandDesc bd = operand_desc(sB(s), 0, C::kBBytes);
          const uint32_t d = tmem + buf * C::BN;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8f6f4_pair(d, ad.base + k * ad.step, bd.base + k * bd.step, idesc,
                            k != 0 ? 1u : 0u);
          mma_commit_pair(empty_bar(s), (uint16_t)0x3);
          mma_commit_pair(accf_bar(buf), (uint16_t)0x3);
        }
      }
      if (!ok) {
        mma_commit_pair(drain_bar, (uint16_t)0x1);
        drain_wait(drain_bar, 0);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------- promotion epilogue (both)
    constexpr int kCols = C::kCols;
    const uint32_t q = warp & 3u;                 // TMEM lane quadrant of this warp
    const int col0 = ((int)(warp - 2) >> 2) * kCols;  // its columns of the BN-wide tile
    const uint32_t lane_base = tmem + ((32u * q) << 16) + (uint32_t)col0;
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
    const int64_t G = args.K / 128;
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = pair; t < num_tiles && ok; t += npairs) {
      const TileInfo ti = tile_info(t);
      const int64_t n0 = ti.n0;
      const int64_t row = ti.m0 + rank * C::BM + 32 * q + lane;
      // this warp's columns lie in one 128-row block of B; a warp wholly
      // past N (or a lane past its rows: past M, or in the next expert's)
      // multiplies by a zero scale and stores nothing
      const bool row_in = row < ti.row_end, cols_in = n0 + col0 < args.N;
      // scale of slice k: sa[k][row] * sb[block][k]; the next slice's pair
      // is loaded one slice ahead, and the line four slices ahead is
      // brought into L2 meanwhile (no registers held for it)
      const float *sa_p = static_cast<const float *>(args.sa) + (row_in ? row : 0);
      const float *sb_p = static_cast<const float *>(args.sb) + ti.sbo + ((n0 + col0) >> 7) * G;
      constexpr int kAhead = 4;
      float na = row_in ? __ldg(sa_p) : 0.0f, nb = cols_in ? __ldg(sb_p) : 0.0f;
      float acc[kCols];
#pragma unroll
      for (int i = 0; i < kCols; ++i) acc[i] = 0.0f;
      for (int k = 0; k < kb_count; ++k) {
        const uint32_t buf = it % C::kAccBufs, use = it / C::kAccBufs;
        const float s_cur = na * nb;
        if (k + 1 < kb_count) {
          sa_p += args.M;
          ++sb_p;
          na = row_in ? __ldg(sa_p) : 0.0f;
          nb = cols_in ? __ldg(sb_p) : 0.0f;
          if (k + kAhead < kb_count) {
            if (row_in) prefetch_l2(sa_p + (kAhead - 1) * args.M);
            if (cols_in && lane == 0) prefetch_l2(sb_p + (kAhead - 1));
          }
        }
        if (!mbar_wait_warp(accf_bar(buf), use & 1u, abort_flag, err, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = lane_base + buf * C::BN;
        // 16-column chunks: chunk c + 1's read is in flight while chunk c's
        // FMAs issue (tcgen05.wait::ld waits for every read of the thread, so
        // one read overlaps the arithmetic at a time); the buffer goes back
        // once the last chunk is read, before its FMAs.  A relaxed arrival:
        // every lane's reads are complete (wait::ld), and a release would
        // first wait for this thread's scale loads and stores in flight.
        constexpr int kC16 = kCols / 16;
        uint32_t r[2][16];
        FP8K_TMEM_LD_X16(tb, r[0]);
#pragma unroll
        for (int c = 0; c < kC16; ++c) {
          tmem_ld_wait();
          FP8K_REG_FENCE16(r[c & 1]);
          if (c + 1 < kC16) {
            FP8K_TMEM_LD_X16(tb + 16 * (c + 1), r[(c + 1) & 1]);
          } else {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acce_leader0 + 8u * buf);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i)
            acc[16 * c + i] = fmaf(s_cur, __uint_as_float(r[c & 1][i]), acc[16 * c + i]);
        }
        ++it;
      }
      if (!ok) break;
      // the tile's origin once more (not held in registers across the slices)
      const TileInfo to = tile_info(t);
      const int64_t orow = to.m0 + rank * C::BM + 32 * q + lane;
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = acc[32 * c + i];
        // (store_row32 itself skips rows past M; expert rows end earlier)
        if (!EXPERTS || orow < to.row_end) store_row32(args, orow, to.n0 + col0 + 32 * c, v);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) tmem_dealloc_pair(tmem, C::kTmemCols);
}

// 256 x 256 pair tiles: six stages of 32 KB, two 256-column TMEM buffers,
// eight epilogue warps (two per TMEM lane quadrant) of 128 columns.  The
// promotion reads every slice's fp32 partial out of TMEM, 4 B per output
// element and 128-deep K group; at the rate these reads reach (about 128 B
// per cycle and SM in every layout measured) that takes 4 BN cycles per
// slice against the tensor core's 2.5 BN, so the kernel tops out near 62% of
// the dense FP8 rate whatever the tile shape.  Measured at 4096 x 2048 x
// 7168 (2 rounds of tiles) / 16384 x 2048 x 7168 (7 rounds):
//   - 256 x 128, eight 64-column warps: 78.5 / 248 us (each CTA's tensor
//     core also reads 8 KB of shared memory, A and both halves of B, per
//     128 x 128 x 32 MMA: its own limit at the same ~62%);
//   - 256 x 256, eight 128-column warps, 16-column reads with the next one
//     in flight under the FMAs: 68.3 / 214 us (this one);
//   - the same with 32-column reads one at a time: 94.8 / 304 us;
//   - 256 x 192, twelve 64-column warps (128 registers): 86.7 / 265 us.
constexpr int kPromoteBN = 256;
constexpr int kPromoteStages = 6;
constexpr int kPromoteEpiWarps = 8;
using PromoteC = PromoteCfg<kPromoteBN, kPromoteStages, kPromoteEpiWarps>;

int gemm_pair_promote_b_rows() { return PromoteC::BN / 2; }

// The pair kernel has no split K: it pays off once the 256 x 256 tiles give
// at least half of the pairs work (one round of them then takes less time
// than the one-CTA kernel's two rounds of 128 x 128 tiles).  K-major
// operands only (the group scales run along K).  Expert-grouped rows count
// the tiles of the rows alone (at most one partial row tile per expert
// more).
bool gemm_pair_promote_eligible(int64_t M, int64_t N, int64_t K, int sms) {
  if (K % 128 != 0) return false;
  const int64_t tiles = ((M + 255) / 256) * ((N + PromoteC::BN - 1) / PromoteC::BN);
  return tiles >= sms / 4;
}

template <bool EXPERTS>
static cudaError_t run_pair_promote(const CUtensorMap &tma, const CUtensorMap &tmb,
                                    const GemmArgs &args, int sms, cudaStream_t st) {
  using C = PromoteC;
  auto kern = gemm_pair_promote_kernel<kPromoteBN, kPromoteStages, kPromoteEpiWarps, EXPERTS>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  // (expert-grouped rows: the tile count is known on the device only; the
  // bound adds one partial row tile per expert)
  const int64_t row_tiles = (args.M + 255) / 256 + (EXPERTS ? args.experts : 0);
  const int64_t tiles = row_tiles * ((args.N + C::BN - 1) / C::BN);
  const int64_t pairs = tiles < sms / 2 ? tiles : sms / 2;
  kern<<<(unsigned)(2 * pairs), C::kThreads, C::kSmem, st>>>(tma, tmb, args);
  return cudaGetLastError();
}

cudaError_t launch_gemm_pair_promote(const CUtensorMap &tma, const CUtensorMap &tmb,
                                     const GemmArgs &args, int sms, cudaStream_t st) {
  if (args.K % 128 != 0 || args.a_mn || args.b_mn || args.ksplit != 1) return cudaErrorInvalidValue;
  if (args.experts > 0) {
    if (args.experts > kMaxExperts || args.offsets == nullptr) return cudaErrorInvalidValue;
    return run_pair_promote<true>(tma, tmb, args, sms, st);
  }
  return run_pair_promote<false>(tma, tmb, args, sms, st);
}

}  // namespace fp8k
