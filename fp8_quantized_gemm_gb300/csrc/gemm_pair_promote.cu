// Per-K-group GEMM with FP32 scales (Transformers fine-grained FP8, 一:
// C[m, n] = sum over 128-wide K groups g of sa[m, g] * sb[n / 128, g] *
// sum_{k in g} qa[m, k] qb[n, k]) on CTA pairs (tcgen05 cta_group::2).
//
// FP32 scales are not powers of two, so the tensor core cannot apply them:
// every 128-deep K slice is contracted into its own TMEM buffer and the
// epilogue warps promote it, acc += sa * sb * partial, in registers.  On one
// CTA with 128 x 128 tiles every k block moves 32 KB through shared memory
// (16 KB of A, 16 KB of B, written by TMA and read by the tensor core) for
// 4.2 MFLOP.  Here two CTAs on neighbouring SMs compute one 256 x 128 tile
// with M = 256 MMAs issued by the even CTA (the leader):
//
//   - each CTA stages its own 128 rows of A and its own 64 rows of B per k
//     block (24 KB a stage, eight stages), both CTAs' copies completing on
//     the leader's full barrier;
//   - the leader's MMAs read both CTAs' shared memory at the same offsets
//     and write each CTA's 128 rows of the slice's partial product into that
//     CTA's TMEM, one of four 128-column buffers in a ring;
//   - tcgen05.commit multicasts each stage release and each "slice ready" to
//     both CTAs; eight epilogue warps per CTA (two per TMEM lane quadrant,
//     64 columns each) read the slice out, hand the buffer back on the
//     leader's barrier (a relaxed arrive: a release one would first wait
//     for the warp's scale prefetches in flight) and then promote it, so
//     the tensor core runs the next slices meanwhile.
//
// The promotion FMAs, 64 per warp and slice, bound the kernel: without them
// the same launch runs about a quarter faster.
//
// The scales of a slice are loaded four slices ahead of its promotion.  The
// 128-wide column tile lies inside one 128-row block of B, so one sb value
// covers the whole tile for a slice.
#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace fp8k {

// 256-row tiles per band of the grouped tile order.
constexpr int64_t kPromoteBandRows = 8;

template <int STAGES, int EPI>
struct PromoteCfg {
  static constexpr int BM = 128, BN = 128, BK = 128;  // per CTA: 128 rows; pair: 256 x 128
  // EPI epilogue warps, EPI / 4 per TMEM lane quadrant, each promoting
  // kCols columns of its 32 rows
  static constexpr int kEpiWarps = EPI;
  static constexpr int kCols = 4 * BN / EPI;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr uint32_t kABytes = BM * BK;
  static constexpr uint32_t kBBytes = (BN / 2) * BK;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTileBytes = STAGES * kStageBytes;
  static constexpr int kAccBufs = 4;
  static constexpr uint32_t kTmemCols = kAccBufs * BN;
  static constexpr int kNumBars = 2 * STAGES + 2 * kAccBufs + 1;
  static constexpr uint32_t kSmem = 1024 + kTileBytes + 8 * kNumBars + 16;
  static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
  static_assert(kTmemCols <= 512, "TMEM budget");
  static_assert(kSmem <= 227 * 1024, "shared-memory budget");
  static_assert(EPI % 4 == 0 && kCols % 32 == 0, "whole 32-column chunks per warp");
};

template <int STAGES, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PromoteCfg<STAGES, EPI>::kThreads, 1)
    gemm_pair_promote_kernel(const __grid_constant__ CUtensorMap tma,
                             const __grid_constant__ CUtensorMap tmb, const GemmArgs args) {
  using C = PromoteCfg<STAGES, EPI>;
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
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barrier inits visible to the peer before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // pair p takes tiles p, p + npairs, ... of the grouped order: bands of
  // kPromoteBandRows 256-row tiles walked column by column, so the pairs in
  // flight share A and B blocks in L2
  const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int64_t rows = (args.M + 255) / 256, tiles_n = (args.N + C::BN - 1) / C::BN;
  const int64_t num_tiles = rows * tiles_n;
  const int kb_count = (int)(args.K / C::BK);
  auto tile_origin = [&](int64_t t, int64_t &m0, int64_t &n0) {
    const int64_t band = t / (kPromoteBandRows * tiles_n);
    const int64_t left = rows - band * kPromoteBandRows;
    const int64_t band_rows = left < kPromoteBandRows ? left : kPromoteBandRows;
    const int64_t local = t - band * kPromoteBandRows * tiles_n;
    m0 = (band * kPromoteBandRows + local % band_rows) * 256;
    n0 = (local / band_rows) * C::BN;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint32_t full_leader0 = mapa_shared(full_bar(0), 0);
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = pair; t < num_tiles && ok; t += npairs) {
      int64_t m0, n0;
      tile_origin(t, m0, n0);
      const int32_t am = (int32_t)(m0 + rank * C::BM);
      const int32_t bn = (int32_t)(n0 + rank * (C::BN / 2));
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
    constexpr int kCols = C::kCols, kChunks = kCols / 32;
    const uint32_t q = warp & 3u;                 // TMEM lane quadrant of this warp
    const int col0 = ((int)(warp - 2) >> 2) * kCols;  // its columns of the 128-wide tile
    const uint32_t lane_base = tmem + ((32u * q) << 16) + (uint32_t)col0;
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
    const float *sa = static_cast<const float *>(args.sa);
    const float *sb = static_cast<const float *>(args.sb);
    const int64_t G = args.K / 128;
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = pair; t < num_tiles && ok; t += npairs) {
      int64_t m0, n0;
      tile_origin(t, m0, n0);
      const int64_t row = m0 + rank * C::BM + 32 * q + lane;
      const float *sb_tile = sb + (n0 >> 7) * G;
      float acc[kCols];
#pragma unroll
      for (int i = 0; i < kCols; ++i) acc[i] = 0.0f;
      // scales of slice k sit in register slot k % kQ, loaded kQ slices
      // before the slice is promoted (constant indices: the loop over the
      // slots is unrolled)
      constexpr int kQ = 4;
      float sa_q[kQ], sb_q[kQ];
      auto load_s = [&](int k, float &fa, float &fb) {
        fa = row < args.M ? __ldg(sa + (int64_t)k * args.M + row) : 0.0f;
        fb = __ldg(sb_tile + k);
      };
#pragma unroll
      for (int d = 0; d < kQ; ++d)
        if (d < kb_count) load_s(d, sa_q[d], sb_q[d]);
      for (int kb = 0; kb < kb_count && ok; kb += kQ) {
#pragma unroll
        for (int j = 0; j < kQ; ++j) {
          const int k = kb + j;
          if (k >= kb_count) break;
          const uint32_t buf = it % C::kAccBufs, use = it / C::kAccBufs;
          const float s_cur = sa_q[j] * sb_q[j];
          if (k + kQ < kb_count) load_s(k + kQ, sa_q[j], sb_q[j]);
          if (!mbar_wait_warp(accf_bar(buf), use & 1u, abort_flag, err, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t r[kCols];
#pragma unroll
          for (int c = 0; c < kChunks; ++c) FP8K_TMEM_LD_X32(lane_base + buf * C::BN + 32 * c, (r + 32 * c));
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          // every lane's reads of the buffer are complete (wait::ld): a
          // relaxed arrival hands it back without waiting for this thread's
          // scale prefetches and output stores still in flight
          if (lane == 0) mbar_arrive_cluster_relaxed(acce_leader0 + 8u * buf);
#pragma unroll
          for (int i = 0; i < kCols; ++i) acc[i] = fmaf(s_cur, __uint_as_float(r[i]), acc[i]);
          ++it;
        }
      }
      if (!ok) break;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = acc[32 * c + i];
        store_row32(args, row, n0 + col0 + 32 * c, v);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) tmem_dealloc_pair(tmem, C::kTmemCols);
}

// Eight stages of 24 KB; eight epilogue warps of 64 columns (sixteen of 32
// columns measured slower: their register budget spills).
constexpr int kPromoteStages = 8;
constexpr int kPromoteEpiWarps = 8;
using PromoteC = PromoteCfg<kPromoteStages, kPromoteEpiWarps>;

int gemm_pair_promote_b_rows() { return PromoteC::BN / 2; }

// The pair kernel has no split K: it pays off when the 256 x 128 tiles give
// every pair work.  K-major operands only (the group scales run along K).
bool gemm_pair_promote_eligible(int64_t M, int64_t N, int64_t K, int sms) {
  if (K % 128 != 0) return false;
  const int64_t tiles = ((M + 255) / 256) * ((N + 127) / 128);
  return tiles >= sms / 2;
}

cudaError_t launch_gemm_pair_promote(const CUtensorMap &tma, const CUtensorMap &tmb,
                                     const GemmArgs &args, int sms, cudaStream_t st) {
  using C = PromoteC;
  if (args.K % 128 != 0 || args.a_mn || args.b_mn || args.ksplit != 1 || args.experts != 0)
    return cudaErrorInvalidValue;
  auto kern = gemm_pair_promote_kernel<kPromoteStages, kPromoteEpiWarps>;
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
  const int64_t tiles = ((args.M + 255) / 256) * ((args.N + C::BN - 1) / C::BN);
  const int64_t pairs = tiles < sms / 2 ? tiles : sms / 2;
  kern<<<(unsigned)(2 * pairs), C::kThreads, C::kSmem, st>>>(tma, tmb, args);
  return cudaGetLastError();
}

}  // namespace fp8k
