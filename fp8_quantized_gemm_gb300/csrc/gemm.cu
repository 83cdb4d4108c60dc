// Scaled-FP8 GEMM kernels on the 5th-generation tensor cores (tcgen05).
//
// One CTA computes one 128 x BN output tile from 128-byte K slices of A
// and B.  Operands are K-major (A [M, K], B [N, K]) in every mode; the
// per-tensor mode also takes MN-major ones (A [K, M], B [K, N]: the codes of
// a row-major tensor used transposed), loaded as 128-wide boxes along M or N
// and described to the MMA as MN-major.
//
//   warp 0        TMA producer: A and B tiles (128-byte swizzle) into a ring
//                 of shared-memory stages; for the block-scaled modes also
//                 the scale-factor words of the stage.
//   warp 1        allocates TMEM; one elected thread issues tcgen05.mma
//                 (4 x K=32 per stage) and tcgen05.commit's each stage back
//                 to the producer.
//   warps 2..     epilogue: tcgen05.ld the FP32 accumulator, apply the
//                 scales, convert, store.
//
// Scale placement (the four modes of kernels.h):
//   per tensor   (Flax guide 2.2)  alpha = sa * sb once in the epilogue.
//   two level    (MOSS blog, 4)    E8M0 local factors as block scale factors
//                                  of kind::mxf8f6f4 (one per 1x32 K block,
//                                  scale_vec::1X), FP32 S_a * S_b in the
//                                  epilogue.
//   group UE8M0  (Transformers 七) the per-128 power-of-two scales, replicated
//                                  over the four 1x32 blocks, as block scale
//                                  factors: no promotion at all.
//   group FP32   (Transformers 一) every 128-wide K slice is contracted into
//                                  its own TMEM buffer (4 buffers in a ring);
//                                  the epilogue warps promote
//                                  acc += sa[m,g] * sb[n/128,g] * partial
//                                  while the tensor cores run the next slice.
//   group FP32, (32, 32) blocks (Transformers 八: weight_block_size (32, 32),
//                                  四: float scales) the same with every K=32
//                                  MMA in its own buffer: a promotion per
//                                  32-deep K step, with the scales of each
//                                  32-column weight block.
#include "common.cuh"
#include "expert_tiles.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace fp8k {

constexpr uint32_t pow2_cols(uint32_t c) {
  uint32_t p = 32;
  while (p < c) p <<= 1;
  return p;
}

// Row tiles per band of the grouped tile order (see tile_info).
constexpr int64_t kBandRows = 16;
// Pipeline depth of the FP32-promotion mode (32 KB stages, no scale-factor
// staging; seven fit beside no expert tables but measured no faster).
constexpr int kF32Stages = 6;

template <int MODE, int BN, int STAGES>
struct Cfg {
  static constexpr int BM = 128, BK = 128;
  static constexpr bool kBlockScaled = (MODE == kScaleMx || MODE == kScaleGroupUe8m0);
  static constexpr bool kPromote = (MODE == kScaleGroupF32 || MODE == kScaleGroupF32x32);
  // promotion slices per 128-wide K block (one per K=32 MMA with 32-wide groups)
  static constexpr int kSub = MODE == kScaleGroupF32x32 ? 4 : 1;
  static constexpr int kEpiWarps = kPromote ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr uint32_t kABytes = BM * BK, kBBytes = BN * BK;
  static constexpr uint32_t kSfaBytes = kBlockScaled ? BM * 4 : 0;
  static constexpr uint32_t kSfbBytes = kBlockScaled ? BN * 4 : 0;
  static constexpr uint32_t kTileBytes = STAGES * (kABytes + kBBytes);
  static constexpr uint32_t kSfBytes = STAGES * (kSfaBytes + kSfbBytes);
  // TMEM accumulators: per-tensor mode double-buffers whole tiles (epilogue of
  // one tile overlaps the MMAs of the next); the promotion mode rings four
  // per-K-slice buffers; the block-scaled modes keep one tile buffer next to
  // their per-stage scale-factor columns.
  static constexpr int kAccBufs = kPromote ? 4 : (MODE == kScaleTensor ? 2 : 1);
  static constexpr uint32_t kAccCols = kAccBufs * BN;
  static constexpr uint32_t kSfColsPerStage = kBlockScaled ? 4 + BN / 32 : 0;
  static constexpr uint32_t kTmemCols = pow2_cols(kAccCols + STAGES * kSfColsPerStage);
  static constexpr int kNumBars = 2 * STAGES + 2 * kAccBufs + 1;  // + drain
  static constexpr uint32_t kSmem = 1024 + kTileBytes + kSfBytes + 8 * kNumBars + 16;
  static_assert(kTmemCols <= 512, "TMEM budget");
  static_assert(kSmem <= 227 * 1024, "shared-memory budget");
  static_assert(BN % 32 == 0 && BN <= 256, "tile N");
};

// Epilogue factor of the block-scaled mode: the two global factors, or 1
// when there are none (per-row factors, or UE8M0 group scales run as E8M0
// words).
__device__ __forceinline__ float mx_alpha(const GemmArgs &a) {
  return a.row_scale != nullptr || a.ga == nullptr ? 1.0f : *a.ga * *a.gb;
}

// MC == 2: the two CTAs of a cluster take vertically adjacent tiles (row
// tiles 2p and 2p + 1, the same columns) and share the B box of every stage:
// each CTA loads one half of it and multicasts that half to both, so the L2
// traffic of B halves; a stage is refilled once both CTAs' MMAs have
// released it (the commit arrives on both CTAs' empty barriers).
template <int MODE, int BN, int STAGES, bool EXPERTS, int MC>
__global__ void __launch_bounds__(Cfg<MODE, BN, STAGES>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                const GemmArgs args) {
  using C = Cfg<MODE, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *tiles = smem;
  uint8_t *sf = smem + C::kTileBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sf + C::kSfBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const DevErr err{args.err, args.wait_limit_ns};
  // split cluster: after the main loop the stage buffers hold this split's
  // fp32 partial tile, [128][kPartStride] (see cluster_reduce)
  float *part = reinterpret_cast<float *>(tiles);
  static_assert((uint32_t)C::BM * kPartStride<BN> * 4 <= C::kTileBytes, "partial tile fits the stages");

  auto sA = [&](int s) { return smem_u32(tiles + s * (C::kABytes + C::kBBytes)); };
  auto sB = [&](int s) { return smem_u32(tiles + s * (C::kABytes + C::kBBytes) + C::kABytes); };
  auto sSfa = [&](int s) { return sf + s * (C::kSfaBytes + C::kSfbBytes); };
  auto sSfb = [&](int s) { return sf + s * (C::kSfaBytes + C::kSfbBytes) + C::kSfaBytes; };
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
  auto accf_bar = [&](int b) { return smem_u32(&bars[2 * STAGES + b]); };
  auto acce_bar = [&](int b) { return smem_u32(&bars[2 * STAGES + C::kAccBufs + b]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * STAGES + 2 * C::kAccBufs]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), MC);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), C::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma);
    tma_prefetch_desc(&tmb);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Programmatic dependent launch: the next kernel may start now; this one
  // reads nothing a previous kernel may write (the expert offsets, the
  // operands, the scales) and writes nothing before grid_dependency_wait()
  // below (the grouped-expert kernels wait here, before their table).
  launch_dependents();
  if constexpr (EXPERTS) grid_dependency_wait();

  // Persistent tile loop: tile t covers rows (t / tiles_n) * 128 and columns
  // (t % tiles_n) * BN; CTA b takes tiles b, b + gridDim.x, ...  Consecutive
  // CTAs share an A row block (L2 reuse of A; B is read by every row block).
  const int64_t tiles_n = (args.N + BN - 1) / BN;
  // Expert-grouped rows: a tile never spans two experts; expert e owns
  // ceil(rows_e / 128) * tiles_n consecutive tile indices (expert_tiles.cuh).
  // The plain kernels keep no table (EXPERTS false).
  __shared__ ExpertTiles<EXPERTS> ex;
  const int E = EXPERTS ? args.experts : 0;
  if constexpr (EXPERTS) {
    if (warp == 0) build_expert_tiles(args.offsets, E, args.M, tiles_n, C::BM, lane, ex);
    __syncthreads();
  }
  static_assert(MC == 1 || (MC == 2 && !EXPERTS), "multicast pairs plain row tiles");
  const int64_t row_tiles = (args.M + C::BM - 1) / C::BM;
  const int64_t num_tiles =
      EXPERTS ? ex.tile0[E] : (MC == 2 ? (row_tiles + 1) / 2 : row_tiles) * tiles_n;
  const uint32_t mc_rank = MC == 2 ? cluster_ctarank() : 0u;
  const int KB = (int)((args.K + C::BK - 1) / C::BK);
  // work unit u = (tile u % num_tiles, K split u / num_tiles); with ksplit 1
  // units are tiles.  Split s covers k blocks [s*KB/ks, (s+1)*KB/ks).
  const int ks = args.ksplit;
  const int64_t num_units = num_tiles * ks;
  // Tile origin: rows [m0, row_end) of A and C (row_end ends the expert's
  // rows), columns [n0, n0 + BN), B tensor-map row brow, scale offset sbo,
  // and (expert-grouped rows) the row tile's index in the list of all
  // experts' row tiles (atile: the block-scaled mode's per-tile A words).
  struct TileInfo {
    int64_t m0, n0, row_end, brow, sbo, atile;
  };
  auto tile_info = [&](int64_t t) {
    TileInfo ti;
    if constexpr (EXPERTS) {
      const int lo = expert_of_tile(ex, E, t);
      const int64_t local = t - ex.tile0[lo];
      ti.m0 = ex.row0[lo] + (local / tiles_n) * C::BM;
      ti.n0 = (local % tiles_n) * BN;
      ti.row_end = ex.row0[lo + 1];
      ti.brow = (int64_t)lo * args.N + ti.n0;
      ti.sbo = (int64_t)lo * args.sb_expert_stride;
      ti.atile = ex.tile0[lo] / tiles_n + local / tiles_n;
    } else {
      // Grouped order: bands of kBandRows row tiles (row-tile pairs when
      // MC == 2), each walked column by column, so the CTAs in flight share
      // a few A row blocks and B column blocks and both stay in L2 (a plain
      // row-major order streams all of B once per wave of row blocks).
      const int64_t rows = MC == 2 ? (row_tiles + 1) / 2 : row_tiles;
      const int64_t band = t / (kBandRows * tiles_n);
      const int64_t band_rows =
          rows - band * kBandRows < kBandRows ? rows - band * kBandRows : kBandRows;
      const int64_t local = t - band * kBandRows * tiles_n;
      const int64_t mt = band * kBandRows + local % band_rows;
      // (MC == 2: mt indexes row-tile pairs; this CTA takes row tile 2 mt + rank)
      ti.m0 = (mt * MC + mc_rank) * C::BM;
      ti.n0 = (local / band_rows) * BN;
      ti.row_end = args.M;
      ti.brow = ti.n0;
      ti.sbo = 0;
      ti.atile = 0;
    }
    return ti;
  };
  // the CTA's units: u_first, u_first + u_step, ...  In a split cluster the
  // CTA owns exactly one unit: tile = cluster index, split = cluster rank.
  const bool csplit = args.cluster_split != 0;
  const int64_t u_first = csplit ? (int64_t)cluster_ctarank() * num_tiles + blockIdx.x / ks
                                 : (int64_t)(blockIdx.x / MC);
  const int64_t u_step = csplit ? num_units : (int64_t)(gridDim.x / MC);
  auto unit_tile = [&](int64_t u) { return u % num_tiles; };
  auto kb_begin = [&](int64_t u) { return (int)((u / num_tiles) * KB / ks); };
  auto kb_end = [&](int64_t u) { return (int)((u / num_tiles + 1) * KB / ks); };

  if constexpr (!EXPERTS) {
    // the first unit's weight boxes into L2 while the previous kernel may
    // still run (a cache hint: L2 is the device's point of coherence), then
    // wait for that kernel
    if (warp == 0 && lane == 0 && MC == 1 && !args.b_mn && u_first < num_units) {
      const TileInfo ti = tile_info(unit_tile(u_first));
      const int k0 = kb_begin(u_first), k1 = kb_end(u_first);
      for (int kb = k0; kb < k1 && kb < k0 + STAGES; ++kb)
        tma_prefetch_l2_2d(&tmb, kb * C::BK, (int32_t)ti.brow);
    }
    grid_dependency_wait();
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0;  // stage iterations issued, across tiles
    bool ok = true;
    // group-UE8M0 mode: the per-128 scale bytes of a k block are loaded into
    // registers kSfAhead (= STAGES) k blocks before their stage is filled,
    // so the producer does not wait on scale loads (with a one-deep prefetch
    // every stage paid a load latency, which dominated small-M GEMMs; a
    // queue much deeper than the ring measured slower: the unrolled stage
    // loop below grows with it).  The queue
    // is kSfAhead register slots used round-robin with compile-time indices
    // (the stage loop below is unrolled over the slots), so no register ever
    // moves while its load is still in flight.
    constexpr int kSfAhead = MODE == kScaleGroupUe8m0 ? STAGES : 1;
    uint32_t sfa_q[kSfAhead][4] = {}, sfb_q[kSfAhead][BN / 32] = {};
    // A position in the CTA's flat k-block sequence, with the unit's tile
    // origin and k range cached (64-bit divisions once per unit, not per k
    // block: the producer issues every stage and must stay cheap).
    struct Cursor {
      int64_t u, m0, n0, brow, sbo, atile;
      int kb, kb_end;
    };
    auto enter = [&](Cursor &c, int64_t u) {
      c.u = u;
      if (u < num_units) {
        const TileInfo ti = tile_info(unit_tile(u));
        c.m0 = ti.m0;
        c.n0 = ti.n0;
        c.brow = ti.brow;
        c.sbo = ti.sbo;
        c.atile = ti.atile;
        c.kb = kb_begin(u);
        c.kb_end = kb_end(u);
      }
    };
    auto next_kb = [&](Cursor &c) {
      if (++c.kb >= c.kb_end) enter(c, c.u + u_step);
    };
    auto load_sf = [&](const Cursor &cs, uint32_t (&fa)[4], uint32_t (&fb)[BN / 32]) {
      if constexpr (MODE == kScaleGroupUe8m0) {
        const uint8_t *sa8 = static_cast<const uint8_t *>(args.sa);
        const uint8_t *sb8 = static_cast<const uint8_t *>(args.sb);
        const int64_t G = args.K / 128;
        const int64_t m0 = cs.m0, n0 = cs.n0;
        const int kb = cs.kb;
        sb8 += cs.sbo;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t m = m0 + 32 * c + lane;
          fa[c] = m < args.M ? (uint32_t)__ldg(sa8 + (int64_t)kb * args.M + m) : 127u;
        }
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          const int64_t n = n0 + 32 * c + lane;
          fb[c] = n < args.N ? (uint32_t)__ldg(sb8 + (n >> 7) * G + kb) : 127u;
        }
      }
    };
    // the CTA's k blocks as one flat sequence: `cur` is the one the next
    // stage takes, `look` the one whose scales are loaded next
    Cursor cur, look;
    enter(cur, u_first);
    enter(look, u_first);
    auto push_sf = [&](uint32_t (&fa)[4], uint32_t (&fb)[BN / 32]) {
      if (look.u < num_units) {
        load_sf(look, fa, fb);
        next_kb(look);
      }
    };
    if constexpr (MODE == kScaleGroupUe8m0) {
#pragma unroll
      for (int d = 0; d < kSfAhead; ++d) push_sf(sfa_q[d], sfb_q[d]);
    }
    // one k block (cu, ckb) into stage it % STAGES; false when a wait gave up
    auto stage = [&](uint32_t (&fa)[4], uint32_t (&fb)[BN / 32]) -> bool {
      const int64_t m0 = cur.m0, n0 = cur.n0, brow = cur.brow;
      const int kb = cur.kb;
      const int s = (int)(it % STAGES);
      const uint32_t round = it / STAGES;
      if (!mbar_wait_warp(empty_bar(s), (round & 1u) ^ 1u, abort_flag, err, 1)) return false;
      uint32_t tx = C::kABytes + C::kBBytes;
      if constexpr (MODE == kScaleGroupUe8m0) {
        // byte -> word with the byte in all four 1x32 slots; the word for
        // row 32c + l of a 128-row chunk sits at index 4l + c
        uint32_t *wa = reinterpret_cast<uint32_t *>(sSfa(s));
        uint32_t *wb = reinterpret_cast<uint32_t *>(sSfb(s));
#pragma unroll
        for (int c = 0; c < 4; ++c) wa[4 * lane + c] = fa[c] * 0x01010101u;
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
          wb[(c >> 2) * 128 + 4 * lane + (c & 3)] = fb[c] * 0x01010101u;
        fence_proxy_async_smem();
        __syncwarp();
        push_sf(fa, fb);  // this slot now waits for the k block kSfAhead ahead
      }
      if (elect_one()) {
        uint32_t sfb_bytes = 0;
        // (a multicast CTA whose row tile lies past M loads no A factors)
        const int64_t a_mpad = (args.M + 127) / 128 * 128;
        // block-scaled words: B rows n (or e * N + n with experts) of the
        // [K/128][rows padded to 128] word array
        const int64_t b_rows = EXPERTS ? (int64_t)args.experts * args.N : args.N;
        const int64_t b_npad = (b_rows + 127) / 128 * 128;
        const bool a_words = EXPERTS || m0 < a_mpad;
        if constexpr (MODE == kScaleMx) {
          const int64_t rows = (b_npad - brow) < BN ? (b_npad - brow) : BN;
          sfb_bytes = (uint32_t)rows * 4u;
          tx += (a_words ? C::kSfaBytes : 0u) + sfb_bytes;
        }
        mbar_arrive_expect_tx(full_bar(s), tx);
        // tensor-map coordinates are (contiguous dim, row); an MN-major
        // operand is loaded as 128-wide boxes along M or N, 16 KB apart
        const int32_t k0 = kb * C::BK;
        if (args.a_mn)
          tma_load_2d(sA(s), &tma, full_bar(s), (int32_t)m0, k0);
        else
          tma_load_2d(sA(s), &tma, full_bar(s), k0, (int32_t)m0);
        if constexpr (MC == 2) {
          // this CTA's half of the B box (tensor-map box BN / 2 rows), to both
          tma_load_2d_mc(sB(s) + mc_rank * (BN / 2) * C::BK, &tmb, full_bar(s), k0,
                         (int32_t)brow + (int32_t)mc_rank * (BN / 2), (uint16_t)0x3);
        } else if (args.b_mn) {
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            tma_load_2d(sB(s) + h * 128 * C::BK, &tmb, full_bar(s), (int32_t)n0 + 128 * h, k0);
        } else {
          tma_load_2d(sB(s), &tmb, full_bar(s), k0, (int32_t)brow);
        }
        if constexpr (MODE == kScaleMx) {
          // A words: [K/128][M padded] by row, or with experts per row tile,
          // [tile][K/128][128]
          const uint32_t *la = static_cast<const uint32_t *>(args.sa) +
                               (EXPERTS ? (cur.atile * KB + kb) * 128 : (int64_t)kb * a_mpad + m0);
          const uint32_t *lb = static_cast<const uint32_t *>(args.sb) + (int64_t)kb * b_npad + brow;
          if (a_words) bulk_load(smem_u32(sSfa(s)), la, C::kSfaBytes, full_bar(s));
          bulk_load(smem_u32(sSfb(s)), lb, sfb_bytes, full_bar(s));
        }
      }
      __syncwarp();
      ++it;
      next_kb(cur);
      return true;
    };
    while (cur.u < num_units && ok) {
#pragma unroll
      for (int j = 0; j < kSfAhead; ++j) {
        if (cur.u >= num_units || !ok) break;
        ok = stage(sfa_q[j], sfb_q[j]);
      }
    }
    if (!ok && lane == 0) {
      // let the copies already in flight land before the CTA can exit
      const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
      for (uint32_t i = first; i < it; ++i) drain_wait(full_bar(i % STAGES), (i / STAGES) & 1u);
      // the peer's multicast halves for stages this CTA never armed
      if (MC == 2) grace_wait(20000000ull);  // 20 ms
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (elect_one()) {
      uint32_t it = 0, j = 0;
      bool ok = true;
      for (int64_t u = u_first; u < num_units && ok; u += u_step, ++j) {
        uint32_t d = tmem;
        const int kb0 = kb_begin(u), kb1 = kb_end(u);
        uint32_t tile_buf = 0;
        if constexpr (!C::kPromote) {
          tile_buf = j % C::kAccBufs;
          const uint32_t use = j / C::kAccBufs;
          if (!mbar_wait(acce_bar(tile_buf), (use & 1u) ^ 1u, abort_flag, err, 2)) {
            ok = false;
            break;
          }
          d = tmem + tile_buf * BN;
        }
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = (int)(it % STAGES);
          const uint32_t round = it / STAGES;
          if (!mbar_wait(full_bar(s), round & 1u, abort_flag, err, 2)) {
            ok = false;
            break;
          }
          if constexpr (MODE == kScaleGroupF32x32) {
            // every K=32 MMA into its own TMEM buffer (four in a ring), each
            // committed to the epilogue as soon as it is issued
            tc_fence_after();
            const uint32_t idesc = idesc_f8f6f4(128, BN, args.fa, args.fb, 0, 0);
            const OperandDesc ad = operand_desc(sA(s), 0, C::kABytes);
            const OperandDesc bd = operand_desc(sB(s), 0, 128 * C::BK);
#pragma unroll 1
            for (int k = 0; k < 4 && ok; ++k) {
              const uint32_t sub = it * 4u + (uint32_t)k, buf = sub & 3u, use = sub >> 2;
              if (!mbar_wait(acce_bar(buf), (use & 1u) ^ 1u, abort_flag, err, 2)) {
                ok = false;
                break;
              }
              tc_fence_after();
              mma_f8f6f4(tmem + buf * BN, ad.base + k * ad.step, bd.base + k * bd.step, idesc, 0u);
              mma_commit(accf_bar(buf));
            }
            if (!ok) break;
            mma_commit(empty_bar(s));
            continue;
          }
          if constexpr (C::kPromote) {
            // one TMEM buffer per 128-wide K slice, four in a ring
            const uint32_t buf = it & 3u, use = it >> 2;
            if (!mbar_wait(acce_bar(buf), (use & 1u) ^ 1u, abort_flag, err, 2)) {
              ok = false;
              break;
            }
            d = tmem + buf * BN;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_sw128(sA(s));
          const uint64_t bdesc = sdesc_sw128(sB(s));
          if constexpr (C::kBlockScaled) {
            const uint32_t sfa_col = C::kAccCols + (uint32_t)s * C::kSfColsPerStage;
            const uint32_t sfb_col = sfa_col + 4;
            tmem_cp_32x128b_warpx4(tmem + sfa_col, sdesc_plain(smem_u32(sSfa(s))));
#pragma unroll
            for (int jj = 0; jj < BN / 128; ++jj)
              tmem_cp_32x128b_warpx4(tmem + sfb_col + 4 * jj,
                                     sdesc_plain(smem_u32(sSfb(s)) + 512 * jj));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t idesc = idesc_mxf8f6f4(128, BN, args.fa, args.fb, k, k);
              mma_mxf8f6f4(d, adesc + 2 * k, bdesc + 2 * k, idesc, tmem + sfa_col,
                           tmem + sfb_col, (kb != kb0 || k != 0) ? 1u : 0u);
            }
          } else {
            const uint32_t idesc = idesc_f8f6f4(128, BN, args.fa, args.fb, args.a_mn, args.b_mn);
            const OperandDesc ad = operand_desc(sA(s), args.a_mn, C::kABytes);
            const OperandDesc bd = operand_desc(sB(s), args.b_mn, 128 * C::BK);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const bool acc = C::kPromote ? (k != 0) : (kb != kb0 || k != 0);
              mma_f8f6f4(d, ad.base + k * ad.step, bd.base + k * bd.step, idesc, acc ? 1u : 0u);
            }
          }
          if constexpr (MC == 2)
            mma_commit_mc(empty_bar(s), (uint16_t)0x3);
          else
            mma_commit(empty_bar(s));
          if constexpr (C::kPromote) mma_commit(accf_bar(it & 3u));
        }
        if (!ok) break;
        if constexpr (!C::kPromote) mma_commit(accf_bar(tile_buf));
      }
      if (!ok) {
        mma_commit(drain_bar);
        drain_wait(drain_bar, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Split-K arrival: every epilogue thread has written (and fenced) its
    // partials; one thread counts the split in; the last of the tile's splits
    // reduces, then resets the counter for the next call.
    __shared__ int split_last;
    auto finish_split = [&](int64_t t) -> bool {
      __threadfence();
      epi_sync<C::kEpiWarps * 32>();
      if (threadIdx.x == 64) {
        const uint32_t old = atomicAdd(args.counters + t, 1u);
        split_last = (old == (uint32_t)(ks - 1));
        if (split_last) args.counters[t] = 0u;
      }
      epi_sync<C::kEpiWarps * 32>();
      const bool last = split_last != 0;
      if (last) __threadfence();
      return last;
    };
    const uint32_t q = warp & 3u;
    const uint32_t lane_base = tmem + ((32u * q) << 16);
    if constexpr (!C::kPromote) {
      float alpha = 1.0f;
      if constexpr (MODE == kScaleTensor)
        alpha = *static_cast<const float *>(args.sa) * *static_cast<const float *>(args.sb);
      if constexpr (MODE == kScaleMx) alpha = mx_alpha(args);
      uint32_t j = 0;
      for (int64_t u = u_first; u < num_units; u += u_step, ++j) {
        const int64_t t = unit_tile(u);
        const int split = (int)(u / num_tiles);
        const TileInfo ti = tile_info(t);
        const int64_t m0 = ti.m0, n0 = ti.n0;
        // rows past the tile's expert belong to the next expert: not stored
        const int64_t row = m0 + 32 * q + lane < ti.row_end ? m0 + 32 * q + lane : args.M;
        const uint32_t buf = j % C::kAccBufs, use = j / C::kAccBufs;
        const bool got = mbar_wait_warp(accf_bar(buf), use & 1u, abort_flag, err, 3);
        if (ks == 1 && !got) break;
        // split K: every epilogue warp learns whether any gave up before the
        // named barriers of the split arrival
        if (ks > 1 && epi_any<C::kEpiWarps * 32>(!got)) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          FP8K_TMEM_LD_X32(lane_base + buf * BN + (uint32_t)c, r);
          tmem_ld_wait();
          if (c + 32 == BN) {  // accumulator fully read: hand it back to the MMA
            tc_fence_before();
            __syncwarp();
            // (relaxed: the reads are complete; the stores of the earlier
            // chunks need not be)
            if (lane == 0) mbar_arrive_relaxed(acce_bar(buf));
          }
          float v[32];
          if (ks == 1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * alpha;
            store_row32(args, row, n0 + c, v);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
            if (csplit)
              stash_partial32_bn<BN>(part, 32 * q + lane, c, v);
            else
              store_partial32(args, split, row, n0 + c, v);
          }
        }
        if (ks > 1 && !csplit && finish_split(t))
          reduce_split_tile(args, m0, n0, C::BM, BN, alpha, (int)threadIdx.x - 64,
                            C::kEpiWarps * 32);
      }
    } else {
      const int h = (int)(warp - 2) >> 2;  // column half of the 128-wide tile
      const float *sa = static_cast<const float *>(args.sa);
      const float *sb = static_cast<const float *>(args.sb);
      // scale groups along K: 128-wide (one per k block), or 32-wide
      constexpr int kGS = 128 / C::kSub;
      const int64_t G = (args.K + kGS - 1) / kGS;
      const int64_t nb32 = (args.N + 31) / 32;  // 32-row weight blocks
      uint32_t it = 0;
      bool ok = true;
      for (int64_t u = u_first; u < num_units && ok; u += u_step) {
        const int64_t t = unit_tile(u);
        const int split = (int)(u / num_tiles);
        // promotion slices [kb0, kb1): k blocks, or K=32 steps (kSub per block)
        const int kb0 = kb_begin(u) * C::kSub, kb1 = kb_end(u) * C::kSub;
        const TileInfo ti = tile_info(t);
        const int64_t m0 = ti.m0, n0 = ti.n0;
        // rows past the tile's expert belong to the next expert: not stored
        const int64_t row = m0 + 32 * q + lane < ti.row_end ? m0 + 32 * q + lane : args.M;
        // the weight scales of this thread's two 32-column halves: one
        // 128 x 128 block for both, or two 32 x 32 block rows
        const int64_t wb0 = C::kSub == 1 ? (n0 >> 7) : ((n0 + h * 64) >> 5);
        const float *sb_row0 = sb + ti.sbo + (C::kSub == 1 ? wb0 : (wb0 < nb32 ? wb0 : 0)) * G;
        const float *sb_row1 = C::kSub == 1 ? sb_row0 : sb + (wb0 + 1 < nb32 ? wb0 + 1 : 0) * G;
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
        // the scales of a slice are loaded kQ slices before it is promoted,
        // into register slots used round-robin (constant indices: the loop is
        // unrolled over the slots), so no promotion step waits on a scale load
        constexpr int kQ = 4;
        float sa_q[kQ], sb_q[kQ], sb2_q[kQ];
        auto load_s = [&](int k, float &fa, float &fb, float &fb2) {
          fa = row < args.M ? __ldg(sa + (int64_t)k * args.M + row) : 0.0f;
          fb = __ldg(sb_row0 + k);
          fb2 = C::kSub == 1 ? fb : __ldg(sb_row1 + k);
        };
#pragma unroll
        for (int d = 0; d < kQ; ++d)
          if (kb0 + d < kb1) load_s(kb0 + d, sa_q[d], sb_q[d], sb2_q[d]);
        for (int kb = kb0; kb < kb1 && ok; kb += kQ) {
#pragma unroll
          for (int j = 0; j < kQ; ++j) {
            const int k = kb + j;
            if (k >= kb1) break;
            const uint32_t buf = it & 3u, use = it >> 2;
            const float s_cur = sa_q[j] * sb_q[j];
            const float s_cur2 = sa_q[j] * sb2_q[j];
            if (k + kQ < kb1) load_s(k + kQ, sa_q[j], sb_q[j], sb2_q[j]);
            if (!mbar_wait_warp(accf_bar(buf), use & 1u, abort_flag, err, 3)) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint32_t r0[32], r1[32];
            const uint32_t col = buf * BN + (uint32_t)(h * 64);
            FP8K_TMEM_LD_X32(lane_base + col, r0);
            FP8K_TMEM_LD_X32(lane_base + col + 32, r1);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            // the reads are complete (wait::ld): a relaxed arrival hands the
            // buffer back without waiting for the scale prefetches in flight
            if (lane == 0) mbar_arrive_relaxed(acce_bar(buf));
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              acc[i] = fmaf(s_cur, __uint_as_float(r0[i]), acc[i]);
              acc[32 + i] = fmaf(s_cur2, __uint_as_float(r1[i]), acc[32 + i]);
            }
            ++it;
          }
        }
        if (ks == 1 && !ok) break;
        if (ks > 1 && epi_any<C::kEpiWarps * 32>(!ok)) break;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = acc[i];
        if (ks == 1) store_row32(args, row, n0 + h * 64, v);
        else if (csplit) stash_partial32_bn<BN>(part, 32 * q + lane, h * 64, v);
        else store_partial32(args, split, row, n0 + h * 64, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = acc[32 + i];
        if (ks == 1) store_row32(args, row, n0 + h * 64 + 32, v);
        else if (csplit) stash_partial32_bn<BN>(part, 32 * q + lane, h * 64 + 32, v);
        else store_partial32(args, split, row, n0 + h * 64 + 32, v);
        if (ks > 1 && !csplit && finish_split(t))
          reduce_split_tile(args, m0, n0, C::BM, BN, 1.0f, (int)threadIdx.x - 64,
                            C::kEpiWarps * 32);
      }
    }
  }

  if (csplit) {
    // every split's partial tile is in its CTA's shared memory: each CTA sums
    // a slice of the tile's rows over the cluster, in split order
    cluster_sync();
    {  // every warp takes part (the producer and MMA warps are done)
      const TileInfo ti = tile_info(unit_tile(u_first));
      const int64_t m0 = ti.m0, n0 = ti.n0;
      float alpha = 1.0f;
      if constexpr (MODE == kScaleTensor)
        alpha = *static_cast<const float *>(args.sa) * *static_cast<const float *>(args.sb);
      if constexpr (MODE == kScaleMx) alpha = mx_alpha(args);
      cluster_reduce<BN>(args, part, m0, n0, C::BM, alpha, cluster_ctarank(), ks,
                         (int)threadIdx.x, C::kThreads);
    }
    cluster_sync();  // no CTA leaves while a peer may still read its partial
  }
  tc_fence_before();
  __syncthreads();
  // a multicast pair leaves together: no CTA exits while the other may still
  // write into its shared memory
  if constexpr (MC == 2) cluster_sync();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// Clusters of `size` CTAs of a GEMM kernel variant that can be resident at
// once.
template <int MODE, int BN, int STAGES, int MC = 1>
static int active_clusters(int size) {
  using C = Cfg<MODE, BN, STAGES>;
  auto kern = gemm_kernel<MODE, BN, STAGES, false, MC>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)size);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess ? n : 0;
}

template <int MODE, int BN, int STAGES, bool EXPERTS = false, int MC = 1>
static cudaError_t run(const CUtensorMap &tma, const CUtensorMap &tmb, const GemmArgs &args,
                       int sms, cudaStream_t st) {
  using C = Cfg<MODE, BN, STAGES>;
  auto kern = gemm_kernel<MODE, BN, STAGES, EXPERTS, MC>;
  if (EXPERTS != (args.experts > 0)) return cudaErrorInvalidValue;
  if (MC == 2 && (args.ksplit != 1 || args.cluster_split || args.b_mn)) return cudaErrorInvalidValue;
  // the shared-memory opt-in is set once per device (not inside a capture)
  static bool attr_done[64] = {};
  static int mc_clusters[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    if (MC == 2) mc_clusters[dev] = active_clusters<MODE, BN, STAGES, MC>(2);
    attr_done[dev] = true;
  }
  // (expert-grouped rows: at most one partial row tile per expert more)
  const int64_t row_tiles = (args.M + C::BM - 1) / C::BM + (args.experts > 0 ? args.experts : 0);
  const int64_t units = row_tiles * ((args.N + BN - 1) / BN) * args.ksplit;
  // programmatic stream serialization: the kernel waits for the previous one
  // itself (grid_dependency_wait) and may start before it ends
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  if (args.cluster_split || MC == 2) {
    cudaLaunchConfig_t cfg = {};
    unsigned csize = 0;
    if (args.cluster_split) {
      // one CTA per unit; the splits of a tile are one cluster
      if (args.ksplit < 2 || args.ksplit > kMaxClusterSplit) return cudaErrorInvalidValue;
      cfg.gridDim = dim3((unsigned)units);
      csize = (unsigned)args.ksplit;
    } else {
      // persistent multicast pairs: one cluster per pair of row tiles
      const int64_t pair_tiles = (row_tiles + 1) / 2 * ((args.N + BN - 1) / BN);
      const int64_t cap = mc_clusters[dev] > 0 ? mc_clusters[dev] : sms / 2;
      cfg.gridDim = dim3((unsigned)(2 * (pair_tiles < cap ? pair_tiles : cap)));
      csize = 2;
    }
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = csize;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tma, tmb, args);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units < sms ? units : sms));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tma, tmb, args);
}

// Tile width: 128 for the FP32-promotion mode; 256 for the per-tensor mode
// (whose large shapes run on CTA pairs); for the block-scaled modes 256 when
// the 128 x 256 tiles fill the SMs and 128 otherwise (twice the tiles: mid-
// size M then needs no split K, small M splits K over fewer k blocks).
int gemm_tile_n(int mode, int64_t M, int64_t N, int sms) {
  if (mode == kScaleGroupF32 || mode == kScaleGroupF32x32) return 128;
  if (mode == kScaleTensor) return 256;
  const int64_t tiles256 = ((M + 127) / 128) * ((N + 255) / 256);
  return tiles256 < sms ? 128 : 256;
}

// Split K when the tiles cannot fill half the SMs: as many splits as fit the
// SMs, each covering at least four 128-wide K blocks.  Cluster splits reduce
// through distributed shared memory (at most kMaxClusterSplit per tile);
// workspace splits are capped at 512 KB of fp32 partials per tile, which the
// last CTA of the tile sums.
static int max_active_clusters(int mode, int bn, int size) {
  static int cache[64][5][2][kMaxClusterSplit + 1];
  static bool have[64][5][2][kMaxClusterSplit + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int w = bn == 128 ? 0 : 1;
  if (!have[dev][mode][w][size]) {
    int n = 0;
    switch (mode) {
      case kScaleTensor: n = active_clusters<kScaleTensor, 256, 4>(size); break;
      case kScaleMx:
        n = w == 0 ? active_clusters<kScaleMx, 128, 6>(size)
                   : active_clusters<kScaleMx, 256, 4>(size);
        break;
      case kScaleGroupUe8m0:
        n = w == 0 ? active_clusters<kScaleGroupUe8m0, 128, 6>(size)
                   : active_clusters<kScaleGroupUe8m0, 256, 4>(size);
        break;
      case kScaleGroupF32x32: n = active_clusters<kScaleGroupF32x32, 128, kF32Stages>(size); break;
      default: n = active_clusters<kScaleGroupF32, 128, kF32Stages>(size); break;
    }
    cache[dev][mode][w][size] = n;
    have[dev][mode][w][size] = true;
  }
  return cache[dev][mode][w][size];
}

int gemm_ksplit(int mode, int64_t M, int64_t N, int64_t K, int sms, bool cluster) {
  const int64_t bn = gemm_tile_n(mode, M, N, sms);
  const int64_t tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
  const int64_t kb = (K + 127) / 128;
  if (tiles * 2 > sms || kb < 8) return 1;
  int64_t ks = sms / tiles;
  if (ks > kb / 4) ks = kb / 4;
  if (cluster) {
    // the largest split whose clusters (one per tile) are all resident at
    // once: a second wave of clusters would double the time
    if (ks > kMaxClusterSplit) ks = kMaxClusterSplit;
    while (ks > 1 && max_active_clusters(mode, (int)bn, (int)ks) < tiles) --ks;
  } else {
    const int64_t rows = M < 128 ? M : 128;
    const int64_t by_partials = (512 * 1024) / (rows * bn * 4);
    if (ks > by_partials) ks = by_partials;
  }
  return ks < 2 ? 1 : (int)ks;
}

cudaError_t launch_gemm_experts(int mode, int bn, const CUtensorMap &tma, const CUtensorMap &tmb,
                                const GemmArgs &args, int sms, cudaStream_t st) {
  // (six stages: the expert tables take 3 KB of static shared memory)
  if (mode == kScaleGroupF32) return run<kScaleGroupF32, 128, 6, true>(tma, tmb, args, sms, st);
  if (mode == kScaleMx) {
    if (bn == 128) return run<kScaleMx, 128, 6, true>(tma, tmb, args, sms, st);
    return run<kScaleMx, 256, 4, true>(tma, tmb, args, sms, st);
  }
  if (mode != kScaleGroupUe8m0) return cudaErrorInvalidValue;
  if (bn == 128) return run<kScaleGroupUe8m0, 128, 6, true>(tma, tmb, args, sms, st);
  return run<kScaleGroupUe8m0, 256, 4, true>(tma, tmb, args, sms, st);
}

cudaError_t launch_gemm(int mode, const CUtensorMap &tma, const CUtensorMap &tmb,
                        const GemmArgs &args, int sms, cudaStream_t st) {
  const bool mc = args.multicast != 0;
  if (mc && mode == kScaleTensor) return cudaErrorInvalidValue;
  switch (mode) {
    case kScaleTensor: return run<kScaleTensor, 256, 4>(tma, tmb, args, sms, st);
    case kScaleMx:
      if (gemm_tile_n(mode, args.M, args.N, sms) == 128)
        return mc ? run<kScaleMx, 128, 6, false, 2>(tma, tmb, args, sms, st)
                  : run<kScaleMx, 128, 6>(tma, tmb, args, sms, st);
      return mc ? run<kScaleMx, 256, 4, false, 2>(tma, tmb, args, sms, st)
                : run<kScaleMx, 256, 4>(tma, tmb, args, sms, st);
    case kScaleGroupUe8m0:
      if (gemm_tile_n(mode, args.M, args.N, sms) == 128)
        return mc ? run<kScaleGroupUe8m0, 128, 6, false, 2>(tma, tmb, args, sms, st)
                  : run<kScaleGroupUe8m0, 128, 6>(tma, tmb, args, sms, st);
      return mc ? run<kScaleGroupUe8m0, 256, 4, false, 2>(tma, tmb, args, sms, st)
                : run<kScaleGroupUe8m0, 256, 4>(tma, tmb, args, sms, st);
    case kScaleGroupF32:
      return mc ? run<kScaleGroupF32, 128, kF32Stages, false, 2>(tma, tmb, args, sms, st)
                : run<kScaleGroupF32, 128, kF32Stages>(tma, tmb, args, sms, st);
    case kScaleGroupF32x32:
      if (mc) return cudaErrorInvalidValue;
      return run<kScaleGroupF32x32, 128, kF32Stages>(tma, tmb, args, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fp8k
