// Per-tensor scaled-FP8 GEMM on CTA pairs (tcgen05 cta_group::2), for one
// problem or a group of independent problems in one launch.
//
// A cluster of two CTAs on neighbouring SMs computes one 256 x BN output tile
// with M = 256 MMAs issued by the even CTA (the leader):
//
//   - each CTA stages its own 128 rows of A and its own half (BN/2 rows) of B
//     per 128-byte K slice, so a stage is 32 KB instead of 48 KB and six
//     stages fit where four did (more bytes in flight per SM);
//   - both CTAs' TMA loads complete on the LEADER's full barrier (the leader
//     expects the bytes of both), the leader's MMA reads both CTAs' shared
//     memory at the same offsets and writes each CTA's 128 rows of D into that
//     CTA's TMEM;
//   - tcgen05.commit multicasts each stage release and each "accumulator
//     full" to both CTAs; both epilogues hand the accumulator back by arriving
//     on the leader's barrier.
//
// Operands may be K-major ([rows, K]) or MN-major ([K, rows], the codes of a
// row-major tensor used transposed); the tensor map, the TMA coordinates, the
// shared-memory descriptors and the instruction descriptor's major bits
// follow the layout, the data flow is the same.
//
// Two TMEM accumulators per CTA: the epilogue of one tile overlaps the MMAs
// of the next.  Scales are applied once in the epilogue (Flax guide 2.2).
//
// Grouped launch: up to kMaxGroup independent problems (each with its own
// operands, formats, scales and output) share one persistent tile space, the
// problems' tiles laid end to end.  The host orders the problems longest-K
// first so that the strided tile assignment stays balanced.  One launch pays
// the prologue, pipeline fill and tail once for all of them (the Float8
// linear's y, dx and dW GEMMs are independent once their operands are
// quantized).
//
// Two epilogue variants fold the training step's element-wise work into the
// GEMM, so that its inputs are read from TMEM instead of HBM (the epilogue of
// one tile runs while the MMAs of the next fill the other accumulator):
//   - gated SwiGLU (h = x W1^T, u = x W3^T): rank 0 of the pair stages rows
//     of W1 and rank 1 the same rows of W3, so each 256 x 256 accumulator is
//     [h | u] for 128 output columns; the epilogue writes h and u (bf16) and
//     the codes of a = silu(h) u under the delayed scale, and its amax;
//   - AdamW on a weight-gradient GEMM: the fp32 gradient tile updates the
//     parameters, moments and bf16 copy in place and is never stored.
// Both use exactly the arithmetic of the standalone kernels (elementwise.cuh),
// so the results are the same bits.
#include "common.cuh"
#include "elementwise.cuh"
#include "gemm_common.cuh"
#include "kernels.h"
#include "quant_common.cuh"

namespace fp8k {

// 256-row tiles per band of the grouped tile order (see tile_ref); the
// launcher's value (fp8_set_option FP8_OPT_GEMM_BAND_ROWS) is passed in
// PairGroup::band_rows.
constexpr int64_t kPairBandRows = 8;

template <int BN, int STAGES>
struct PairCfg {
  static constexpr int BM = 128, BK = 128;  // rows per CTA (256 per pair)
  static constexpr int kEpiWarps = 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr uint32_t kABytes = BM * BK;
  static constexpr uint32_t kBBytes = (BN / 2) * BK;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTileBytes = STAGES * kStageBytes;
  static constexpr int kAccBufs = 2;
  static constexpr uint32_t kTmemCols = kAccBufs * BN;
  static constexpr int kNumBars = 2 * STAGES + 2 * kAccBufs + 1;
  // TMA-store staging: per epilogue warp two 32-row x 128-byte boxes
  static constexpr uint32_t kOutBox = 32 * 128;
  static constexpr uint32_t kOutBytes = kEpiWarps * 2 * kOutBox;
  static constexpr uint32_t kSmem = 1024 + kTileBytes + kOutBytes + 8 * kNumBars + 16;
  static_assert(kTmemCols <= 512, "TMEM budget");
  static_assert(kSmem <= 227 * 1024, "shared-memory budget");
  static_assert(BM == 128 && BN / 2 == 128, "MN-major tiles: one 128-wide TMA box per operand");
  static_assert(2 * kOutBox >= 32 * 36 * 4, "a warp's AdamW staging buffer fits its two boxes");
};

struct PairGroup {
  CUtensorMap tma[kMaxGroup];
  CUtensorMap tmb[kMaxGroup];
  CUtensorMap tmc[kMaxGroup];   // outputs (problems with args.tma_store)
  CUtensorMap tmb2[kMaxGroup];  // second weight of gated problems
  GemmArgs args[kMaxGroup];
  int64_t tile_begin[kMaxGroup + 1];  // problem i owns tiles [tile_begin[i], tile_begin[i+1])
  int count;
  int64_t band_rows;  // 256-row tiles per band of the tile order
};

// Problem owning global tile t (the group is small: a linear scan).
__device__ __forceinline__ int group_of(const PairGroup &g, int64_t t) {
  int i = 0;
  while (i + 1 < g.count && t >= g.tile_begin[i + 1]) ++i;
  return i;
}

// AdamW on a warp's 32 x 32 gradient chunk (rows row0 .. row0 + 31, columns
// col0 ..), restaged through shared memory so that the parameter traffic is
// coalesced: lane l handles rows 4i + l / 8 and the four columns 4 (l % 8) ..
// of each, so eight lanes cover one 128-byte row segment.  `stage` is the
// warp's 32 x kStageLd fp32 buffer (each lane has already written its own
// row's 32 gradients there).  All 24 loads are issued before any update; p,
// m and v stream (each is read and written once per step).
constexpr int kStageLd = 36;  // row pitch in floats: conflict-free float4 rows
__device__ __forceinline__ void adamw_chunk32(const GemmArgs &a, int64_t row0, int64_t col0,
                                              const float *stage, const AdamwHp &hp,
                                              uint32_t lane) {
  const int rs = (int)(lane >> 3), c4 = (int)(lane & 7) * 4;
  const int64_t col = col0 + c4;
  const bool vec = col + 4 <= a.N;
  float4 pv[8], mv[8], vv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t row = row0 + 4 * i + rs;
    if (vec && row < a.M) {
      const int64_t off = row * a.ldc + col;
      pv[i] = __ldcs(reinterpret_cast<const float4 *>(a.adam_p + off));
      mv[i] = __ldcs(reinterpret_cast<const float4 *>(a.adam_m + off));
      vv[i] = __ldcs(reinterpret_cast<const float4 *>(a.adam_v + off));
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + rs;
    const int64_t row = row0 + r;
    if (row >= a.M || col >= a.N) continue;
    const float4 g = *reinterpret_cast<const float4 *>(stage + r * kStageLd + c4);
    const int64_t off = row * a.ldc + col;
    if (vec) {
      adamw4(pv[i], mv[i], vv[i], g, hp);
      __stcs(reinterpret_cast<float4 *>(a.adam_p + off), pv[i]);
      __stcs(reinterpret_cast<float4 *>(a.adam_m + off), mv[i]);
      __stcs(reinterpret_cast<float4 *>(a.adam_v + off), vv[i]);
      if (a.adam_pb != nullptr)
        __stcs(reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(a.adam_pb) + off),
               f32x4_to_bf16(pv[i]));
    } else {  // the ragged last columns
      const float gg[4] = {g.x, g.y, g.z, g.w};
      for (int e = 0; e < 4 && col + e < a.N; ++e) {
        float pp = a.adam_p[off + e], mm = a.adam_m[off + e], vvv = a.adam_v[off + e];
        adamw1(pp, mm, vvv, gg[e], hp);
        a.adam_p[off + e] = pp;
        a.adam_m[off + e] = mm;
        a.adam_v[off + e] = vvv;
        if (a.adam_pb != nullptr)
          static_cast<__nv_bfloat16 *>(a.adam_pb)[off + e] = __float2bfloat16_rn(pp);
      }
    }
  }
}

// The gated SwiGLU epilogue for 32 columns of one row: h and u (fp32 scaled
// results) are rounded to bf16 and stored, a = bf16(silu(h) u) is divided by
// the delayed scale and cast (the codes fp8_swiglu_forward_quantize would
// give for the stored h and u), and |a| enters the running key.  Full
// chunks only (N % 32 == 0 and 16-byte rows, checked by the host).
template <bool kFast>
__device__ __forceinline__ void gated_row32(const GemmArgs &a, int64_t row, int64_t col0,
                                            const float (&hv)[32], const float (&uv)[32],
                                            const ScaleDiv &d, uint32_t &key) {
  if (row >= a.M || col0 >= a.N) return;
  const int64_t off = row * a.ldc + col0;
  float hb[32], ub[32], ab[32];
  uint32_t hw[16], uw[16], aw[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(hv[2 * i], hv[2 * i + 1]);
    const __nv_bfloat162 u2 = __floats2bfloat162_rn(uv[2 * i], uv[2 * i + 1]);
    hw[i] = *reinterpret_cast<const uint32_t *>(&h2);
    uw[i] = *reinterpret_cast<const uint32_t *>(&u2);
    hb[2 * i] = __uint_as_float(hw[i] << 16);
    hb[2 * i + 1] = __uint_as_float(hw[i] & 0xFFFF0000u);
    ub[2 * i] = __uint_as_float(uw[i] << 16);
    ub[2 * i + 1] = __uint_as_float(uw[i] & 0xFFFF0000u);
  }
  uint4 *hd = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.c) + off);
  uint4 *ud = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.swi_u) + off);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    hd[i] = make_uint4(hw[4 * i], hw[4 * i + 1], hw[4 * i + 2], hw[4 * i + 3]);
    ud[i] = make_uint4(uw[4 * i], uw[4 * i + 1], uw[4 * i + 2], uw[4 * i + 3]);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float a0, a1;
    swiglu_value2(hb[2 * i], hb[2 * i + 1], ub[2 * i], ub[2 * i + 1], a0, a1);
    const __nv_bfloat162 a2 = __floats2bfloat162_rn(a0, a1);
    aw[i] = *reinterpret_cast<const uint32_t *>(&a2);
  }
  uint2 c[4];
  if constexpr (kFast) {
    // quotients of |a| clamped, signs from the bf16 words (quant_bf16x8)
    uint32_t key2 = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 w = make_uint4(aw[4 * j], aw[4 * j + 1], aw[4 * j + 2], aw[4 * j + 3]);
      float y[8];
      bf16x8_quotients(w, d, key2, y);
      c[j] = bf16x8_with_signs(pack8(a.swi_fmt, y), w);
    }
    key = max(key, bf16_key_merge(key2));
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      ab[2 * i] = __uint_as_float(aw[i] << 16);
      ab[2 * i + 1] = __uint_as_float(aw[i] & 0xFFFF0000u);
      key = max(key, max(abs_key(ab[2 * i]), abs_key(ab[2 * i + 1])));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float y[8];
      d.div8<false>(*reinterpret_cast<const float(*)[8]>(ab + 8 * j), y);
      c[j] = pack8(a.swi_fmt, y);
    }
  }
  uint4 *qd = reinterpret_cast<uint4 *>(a.swi_q + off);
  qd[0] = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
  qd[1] = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
}

template <int BN, int STAGES>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<BN, STAGES>::kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ PairGroup grp) {
  using C = PairCfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *out_stage = smem + C::kTileBytes;  // 1024-aligned (kTileBytes is)
  uint64_t *bars = reinterpret_cast<uint64_t *>(out_stage + C::kOutBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const DevErr err{grp.args[0].err, grp.args[0].wait_limit_ns};

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
  if (warp == 0 && lane < (uint32_t)grp.count) {
    tma_prefetch_desc(&grp.tma[lane]);
    tma_prefetch_desc(&grp.tmb[lane]);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barrier inits visible to the peer before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // pair p takes global tiles p, p + npairs, ...; within problem i, local
  // tile t covers rows (t / tiles_n) * 256 (this CTA: + rank * 128) and
  // columns (t % tiles_n) * BN
  const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int64_t num_tiles = grp.tile_begin[grp.count];
  struct TileRef {
    int i;
    int64_t m0, n0;
    int kb_count;
  };
  auto tile_ref = [&](int64_t gt) {
    TileRef r;
    r.i = group_of(grp, gt);
    const GemmArgs &a = grp.args[r.i];
    const int64_t t = gt - grp.tile_begin[r.i];
    // a gated tile covers BN / 2 output columns (h and u of each)
    const int64_t tn = a.gated ? BN / 2 : BN;
    const int64_t tiles_n = (a.N + tn - 1) / tn;
    // grouped order: bands of kPairBandRows 256-row tiles walked column by
    // column, so the pairs in flight share A and B blocks in L2
    const int64_t rows = (a.M + 255) / 256;
    const int64_t bandh = grp.band_rows;
    const int64_t band = t / (bandh * tiles_n);
    const int64_t band_rows = rows - band * bandh < bandh ? rows - band * bandh : bandh;
    const int64_t local = t - band * bandh * tiles_n;
    r.m0 = (band * bandh + local % band_rows) * 256;
    r.n0 = (local / band_rows) * tn;
    r.kb_count = (int)((a.K + C::BK - 1) / C::BK);
    return r;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint32_t full_leader0 = mapa_shared(full_bar(0), 0);
    uint32_t it = 0;
    bool ok = true;
    for (int64_t gt = pair; gt < num_tiles && ok; gt += npairs) {
      const TileRef tr = tile_ref(gt);
      const CUtensorMap *ma = &grp.tma[tr.i];
      // gated: both CTAs stage the same B rows, rank 1 from the second weight
      const bool gated = grp.args[tr.i].gated != 0;
      const CUtensorMap *mb = gated && rank != 0 ? &grp.tmb2[tr.i] : &grp.tmb[tr.i];
      const int64_t m0 = tr.m0 + rank * C::BM;
      const int64_t nb0 = gated ? tr.n0 : tr.n0 + rank * (BN / 2);
      for (int kb = 0; kb < tr.kb_count; ++kb, ++it) {
        const int s = (int)(it % STAGES);
        const uint32_t round = it / STAGES;
        if (!mbar_wait_warp(empty_bar(s), (round & 1u) ^ 1u, abort_flag, err, 1)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          // tensor-map coordinates are (contiguous dim, row): (k, m) for a
          // K-major operand, (m, k) for an MN-major one; both boxes are 16 KB
          const GemmArgs &ga = grp.args[tr.i];
          const int32_t k0 = kb * C::BK;
          const int32_t ax = ga.a_mn ? (int32_t)m0 : k0, ay = ga.a_mn ? k0 : (int32_t)m0;
          const int32_t bx = ga.b_mn ? (int32_t)nb0 : k0, by = ga.b_mn ? k0 : (int32_t)nb0;
          if (leader) {
            mbar_arrive_expect_tx(full_bar(s), 2 * C::kStageBytes);
            tma_load_2d(sA(s), ma, full_bar(s), ax, ay);
            tma_load_2d(sB(s), mb, full_bar(s), bx, by);
          } else {
            const uint32_t fb = full_leader0 + 8u * (uint32_t)s;
            tma_load_2d_pair(sA(s), ma, fb, ax, ay);
            tma_load_2d_pair(sB(s), mb, fb, bx, by);
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
      uint32_t it = 0, j = 0;
      bool ok = true;
      for (int64_t gt = pair; gt < num_tiles && ok; gt += npairs, ++j) {
        const TileRef tr = tile_ref(gt);
        const GemmArgs &ga = grp.args[tr.i];
        const uint32_t idesc = idesc_f8f6f4(256, BN, ga.fa, ga.fb, ga.a_mn, ga.b_mn);
        const uint32_t buf = j & 1u, use = j >> 1;
        if (!mbar_wait(acce_bar(buf), (use & 1u) ^ 1u, abort_flag, err, 2)) {
          ok = false;
          break;
        }
        const uint32_t d = tmem + buf * BN;
        for (int kb = 0; kb < tr.kb_count; ++kb, ++it) {
          const int s = (int)(it % STAGES);
          const uint32_t round = it / STAGES;
          if (!mbar_wait(full_bar(s), round & 1u, abort_flag, err, 2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // per CTA each operand tile is 128 rows wide: one 128-element
          // block along M or N, so the MN-major leading offset is not used
          const OperandDesc ad = operand_desc(sA(s), ga.a_mn, C::kABytes);
          const OperandDesc bd = operand_desc(sB(s), ga.b_mn, C::kBBytes);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8f6f4_pair(d, ad.base + k * ad.step, bd.base + k * bd.step, idesc,
                            (kb | k) != 0 ? 1u : 0u);
          mma_commit_pair(empty_bar(s), (uint16_t)0x3);
        }
        if (!ok) break;
        mma_commit_pair(accf_bar(buf), (uint16_t)0x3);
      }
      if (!ok) {
        mma_commit_pair(drain_bar, (uint16_t)0x1);
        drain_wait(drain_bar, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue (both)
    const uint32_t q = warp & 3u;
    const uint32_t lane_base = tmem + ((32u * q) << 16);
    const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
    const uint64_t out_policy = policy_evict_first();
    uint32_t gkey[kMaxGroup] = {};  // running max |a| of each gated problem
    uint32_t j = 0, out_n = 0;
    for (int64_t gt = pair; gt < num_tiles; gt += npairs, ++j) {
      const TileRef tr = tile_ref(gt);
      const GemmArgs &a = grp.args[tr.i];
      const float alpha = *static_cast<const float *>(a.sa) * *static_cast<const float *>(a.sb);
      const int64_t row = tr.m0 + rank * C::BM + 32 * q + lane;
      const uint32_t buf = j & 1u, use = j >> 1;
      if (!mbar_wait_warp(accf_bar(buf), use & 1u, abort_flag, err, 3)) break;
      tc_fence_after();
      if (a.gated) {
        // columns [0, BN/2) of the accumulator are h, [BN/2, BN) are u
        const float alpha_u = *static_cast<const float *>(a.sa) * *a.swi_sb2;
        const ScaleDiv d(*a.swi_scale);
        uint32_t key = 0;
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t rh[32], ru[32];
          FP8K_TMEM_LD_X32(lane_base + buf * BN + (uint32_t)c, rh);
          FP8K_TMEM_LD_X32(lane_base + buf * BN + (uint32_t)(BN / 2 + c), ru);
          tmem_ld_wait();
          if (c + 32 == BN / 2) {  // accumulator read out: hand it back to the leader
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acce_leader0 + 8u * buf);
          }
          float hv[32], uv[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            hv[i] = __uint_as_float(rh[i]) * alpha;
            uv[i] = __uint_as_float(ru[i]) * alpha_u;
          }
          if (d.fast)
            gated_row32<true>(a, row, tr.n0 + c, hv, uv, d, key);
          else
            gated_row32<false>(a, row, tr.n0 + c, hv, uv, d, key);
        }
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g)
          if (g == tr.i) gkey[g] = max(gkey[g], key);
        continue;
      }
      if (a.adam_p != nullptr) {
        // AdamW on the gradient tile; bias corrections from the step counter
        AdamwHp hp = a.adam_hp;
        float bc1 = 0.0f, bc2 = 0.0f;
        if (lane == 0) {
          const int64_t t = *a.adam_step;
          bc1 = bias_correction(a.adam_b1d, t);
          bc2 = bias_correction(a.adam_b2d, t);
        }
        hp.bc1 = __shfl_sync(0xffffffffu, bc1, 0);
        hp.bc2 = __shfl_sync(0xffffffffu, bc2, 0);
        // this warp's 32 x 32 staging buffer (the TMA-store boxes' space;
        // any bulk store still reading it finishes first)
        float *stage = reinterpret_cast<float *>(out_stage + (warp - 2) * 2 * C::kOutBox);
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        const int64_t row0 = tr.m0 + rank * C::BM + 32 * q;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          FP8K_TMEM_LD_X32(lane_base + buf * BN + (uint32_t)c, r);
          tmem_ld_wait();
          if (c + 32 == BN) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acce_leader0 + 8u * buf);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4 *>(stage + lane * kStageLd + 4 * i) = make_float4(
                __uint_as_float(r[4 * i]) * alpha, __uint_as_float(r[4 * i + 1]) * alpha,
                __uint_as_float(r[4 * i + 2]) * alpha, __uint_as_float(r[4 * i + 3]) * alpha);
          __syncwarp();
          adamw_chunk32(a, row0, tr.n0 + c, stage, hp, lane);
          __syncwarp();  // the buffer is rewritten by the next chunk
        }
        continue;
      }
      if (a.tma_store) {
        // 128-byte column chunks (64 bf16 or 32 fp32 values per row) staged
        // as a 32-row box in this warp's two alternating buffers (128-byte
        // swizzle: 16-byte unit u of row l at l * 128 + (u ^ (l & 7)) * 16)
        // and written by one TMA store each
        const bool f32 = a.out_dt == 0;
        const int cw = f32 ? 32 : 64;
        const int32_t row0 = (int32_t)(tr.m0 + rank * C::BM + 32 * q);
#pragma unroll 1
        for (int c = 0; c < BN; c += cw) {
          uint32_t r[64];
          FP8K_TMEM_LD_X32(lane_base + buf * BN + (uint32_t)c, r);
          if (!f32) FP8K_TMEM_LD_X32(lane_base + buf * BN + (uint32_t)c + 32, (r + 32));
          tmem_ld_wait();
          // (relaxed arrivals: the TMEM reads are complete after wait::ld,
          // and nothing else has to be ordered before the hand-back)
          if (c + cw == BN) {  // accumulator read out: hand it back to the leader
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(acce_leader0 + 8u * buf);
          }
          const int64_t col0 = tr.n0 + c;
          uint32_t packed[32];
          if (f32) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float v = __uint_as_float(r[i]) * alpha;
              if (a.bias != nullptr && col0 + i < a.N) v += __ldg(a.bias + col0 + i);
              packed[i] = __float_as_uint(v);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float v0 = __uint_as_float(r[2 * i]) * alpha, v1 = __uint_as_float(r[2 * i + 1]) * alpha;
              if (a.bias != nullptr) {
                if (col0 + 2 * i < a.N) v0 += __ldg(a.bias + col0 + 2 * i);
                if (col0 + 2 * i + 1 < a.N) v1 += __ldg(a.bias + col0 + 2 * i + 1);
              }
              const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
              packed[i] = *reinterpret_cast<const uint32_t *>(&h);
            }
          }
          // boxes wholly past M or N are not stored (a partial box is
          // clipped by TMA); the buffers alternate per store issued, so the
          // store two back, the last reader of this buffer, has read it
          if (row0 < a.M && col0 < a.N) {
            uint8_t *box = out_stage + ((warp - 2) * 2 + (out_n & 1u)) * C::kOutBox;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4 *>(box + lane * 128 + ((u ^ (lane & 7)) << 4)) = make_uint4(
                  packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d_hint(&grp.tmc[tr.i], smem_u32(box), (int32_t)col0, row0, out_policy);
              bulk_commit();
            }
            ++out_n;
          }
        }
        continue;
      }
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        FP8K_TMEM_LD_X32(lane_base + buf * BN + (uint32_t)c, r);
        tmem_ld_wait();
        if (c + 32 == BN) {  // accumulator read out: hand it back to the leader
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(acce_leader0 + 8u * buf);
        }
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * alpha;
        store_row32(a, row, tr.n0 + c, v);
      }
    }
    // every TMA store has finished reading its box and writing C
    if (lane == 0) bulk_wait_all();
    __syncwarp();
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) {
      if (g < grp.count && grp.args[g].gated) {
        const uint32_t k = warp_max_u32(gkey[g]);
        if (lane == 0 && k != 0u) atomicMax(grp.args[g].swi_amax, k);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal it
  if (warp == 1) tmem_dealloc_pair(tmem, C::kTmemCols);
}

constexpr int kPairBN = 256, kPairStages = 6;

int gemm_pair_b_rows() { return kPairBN / 2; }

int64_t gemm_pair_tiles(int64_t M, int64_t N) {
  return ((M + 255) / 256) * ((N + kPairBN - 1) / kPairBN);
}

// CTA pairs pay off when the 256-row tiles still give every pair work.
bool gemm_pair_eligible(int mode, int64_t M, int64_t N, int sms) {
  if (mode != kScaleTensor) return false;
  return gemm_pair_tiles(M, N) * 4 >= sms / 2;
}

// Tiles of one problem: gated problems cover BN / 2 output columns per tile.
int64_t gemm_pair_tiles_of(const GemmArgs &a) {
  const int64_t tn = a.gated ? kPairBN / 2 : kPairBN;
  return ((a.M + 255) / 256) * ((a.N + tn - 1) / tn);
}

cudaError_t launch_gemm_pair_group(const CUtensorMap *tma, const CUtensorMap *tmb,
                                   const CUtensorMap *tmc, const CUtensorMap *tmb2,
                                   const GemmArgs *args, int count, int sms, cudaStream_t st) {
  using C = PairCfg<kPairBN, kPairStages>;
  if (count < 1 || count > kMaxGroup) return cudaErrorInvalidValue;
  auto kern = gemm_pair_kernel<kPairBN, kPairStages>;
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
  PairGroup g{};
  g.count = count;
  g.band_rows = gemm_pair_band_rows();
  g.tile_begin[0] = 0;
  for (int i = 0; i < count; ++i) {
    g.tma[i] = tma[i];
    g.tmb[i] = tmb[i];
    if (tmc != nullptr) g.tmc[i] = tmc[i];
    if (tmb2 != nullptr) g.tmb2[i] = tmb2[i];
    g.args[i] = args[i];
    if (tmc == nullptr) g.args[i].tma_store = 0;
    if (tmb2 == nullptr) g.args[i].gated = 0;
    if (g.args[i].gated) {  // the fused amax starts from zero
      e = cudaMemsetAsync(g.args[i].swi_amax, 0, sizeof(uint32_t), st);
      if (e != cudaSuccess) return e;
    }
    g.tile_begin[i + 1] = g.tile_begin[i] + gemm_pair_tiles_of(g.args[i]);
  }
  for (int i = count; i < kMaxGroup; ++i) g.tile_begin[i + 1] = g.tile_begin[count];
  const int64_t tiles = g.tile_begin[count];
  const int64_t pairs = tiles < sms / 2 ? tiles : sms / 2;
  kern<<<(unsigned)(2 * pairs), C::kThreads, C::kSmem, st>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_gemm_pair(const CUtensorMap &tma, const CUtensorMap &tmb,
                             const CUtensorMap &tmc, const GemmArgs &args, int sms,
                             cudaStream_t st) {
  return launch_gemm_pair_group(&tma, &tmb, &tmc, nullptr, &args, 1, sms, st);
}

}  // namespace fp8k
