// Per-K-group GEMM for few activation rows (M <= 128), the decode-sized
// shape of fine-grained FP8 (Transformers fine-grained FP8, 一: C[m, n] =
// sum over 128-wide K groups g of sa[m, g] * sb[n / 128, g] *
// sum_{k in g} qa[m, k] qb[n, k]; 六: per-token dynamic activation scales).
//
// At this size the GEMM is a stream over the N x K weight codes, and the
// cost of a launch is its fixed part: the time until every SM has its
// weight bytes in flight, and the time from the last byte to the stored
// result.  So the operands trade places: a CTA's 128 weight rows fill the
// MMA's M side and the activation rows, padded to MP = 16, 32 or 64, its N
// side:
//
//   D[n, m] (TMEM: lane n, column m) = sum_k qb[n0 + n, k] qa[m, k]
//
// The tile's 128 weight rows share one weight-block scale per K group, so
// the promotion after each 128-wide K slice is, per thread (one weight row),
//   acc[m] += (sa[g, m] * sb[n0 / 128, g]) * D[n, m]
// over MP columns only, and each lane fetches the activation scale of one
// column that the warp then shares by shuffles.  65-128 rows run as two
// 64-row halves, a second row of CTAs along the grid's y that streams the
// same weights (its reads hit L2): in CUDA graphs at N 2048, K 7168, M = 128
// took 10.4 / 10.7 us (FP32 / UE8M0 scales) against 11.9 / 13.5 us on the
// general kernel, where one CTA with MP = 128 took 12.6-13.7 us (the
// exchange of a 128 x 128 fp32 partial per CTA, and a stage ring cut to
// four to leave room for its receive buffer).
//
// Each output tile's K range is split over a thread-block cluster of up to
// 8 CTAs (as many as fit beside the other tiles' clusters); each CTA issues
// its k blocks' copies up front (the ring holds most of a CTA's share at K
// 7168).  The reduction is one exchange: CTA r owns weight rows
// [r W, r W + W) of the tile (W = ceil(128 / splits) rounded up to a
// multiple of 4), every CTA stores its partial sums of those rows straight
// into the owner's receive buffer (16-byte remote shared-memory stores,
// which do not wait), one cluster barrier publishes them, and each owner
// sums its rows in split order (the same sums on every run) and stores
// them.  (Staging the partials locally and pushing one bulk copy per owner
// measured no faster.)
//
// Launched with programmatic stream serialization, the kernel overlaps its
// start with the end of the kernel before it: after its setup it asks for
// its own weight boxes to be brought into L2 (a cache hint: L2 is the
// device's point of coherence, so data the previous kernel writes is still
// read correctly), then waits for that kernel to complete before it reads
// or writes anything else, and lets the next kernel start early in turn.
//
//   warp 0   TMA producer: the weight box (128 rows x 128 K) and the
//            activation box (MP rows x 128 K; rows past M read as zero).
//   warp 1   TMEM allocation; one thread issues the 4 x K=32 MMAs of each
//            slice into one of four TMEM buffers (MP columns each).
//   warps 2+ promotion (4 warps, 8 from MP = 32 on: two column halves),
//            then the stores or the exchange.
#include "common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace fp8k {

template <int MP>
struct SkinnyCfg {
  static constexpr uint32_t kWBytes = 128 * 128;  // weight box: 128 rows x 128 K
  static constexpr uint32_t kXBytes = MP * 128;   // activation box
  static constexpr uint32_t kStageBytes = kWBytes + kXBytes;
  // receive buffer of the exchange: [splits][W][kRecvPitch] fp32, one row of
  // MP activation columns per owned weight row (splits * W <= 144 for up to
  // 8 splits); the 16-byte pad puts consecutive rows' vectors in different
  // banks
  static constexpr uint32_t kRecvPitch = MP + 4;
  static constexpr uint32_t kRecvBytes = 144 * kRecvPitch * 4;
  static constexpr uint32_t kBudget = 227 * 1024 - 1024 - kRecvBytes - 512;
  static constexpr int kStages = kBudget / kStageBytes < 8 ? kBudget / kStageBytes : 8;
  static constexpr uint32_t kTileBytes = kStages * kStageBytes;
  static constexpr int kEpiWarps = MP >= 32 ? 8 : 4;
  static constexpr int kCols = MP / (kEpiWarps / 4);  // columns promoted per thread
  static constexpr int kJ = (kCols + 31) / 32;         // scale registers per lane
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kAccBufs = 4;
  static constexpr uint32_t kTmemCols = kAccBufs * MP < 32 ? 32 : kAccBufs * MP;
  static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 1;  // + drain
  static constexpr uint32_t kSmem = 1024 + kTileBytes + kRecvBytes + 8 * kNumBars + 16;
  static_assert(MP == 16 || MP == 32 || MP == 64, "padded activation rows");
  static_assert(kStages >= 4, "pipeline depth");
  static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation");
  static_assert(kSmem <= 227 * 1024, "shared-memory budget");
};

// One group scale as loaded (fp32 bits, or a UE8M0 byte) and as a
// multiplier (2^(b - 127) for a byte).  The loads land in a queue of
// registers and are converted only when used, so no thread waits on a load
// it issued for a later slice.
template <int SFMT>
__device__ __forceinline__ uint32_t skinny_scale_raw(const void *s, int64_t i) {
  if constexpr (SFMT == 0)
    return __float_as_uint(__ldg(static_cast<const float *>(s) + i));
  else
    return (uint32_t)__ldg(static_cast<const uint8_t *>(s) + i);
}
template <int SFMT>
__device__ __forceinline__ float skinny_scale_value(uint32_t raw) {
  if constexpr (SFMT == 0)
    return __uint_as_float(raw);
  else
    return exp2_int((int)raw - 127);
}

template <int SFMT, int MP>
__global__ void __launch_bounds__(SkinnyCfg<MP>::kThreads, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmw,
                       const __grid_constant__ CUtensorMap tmx, const GemmArgs args) {
  using C = SkinnyCfg<MP>;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  if (warp == 0 && lane == 0) {  // descriptor fetches first: the first copies wait on them
    tma_prefetch_desc(&tmw);
    tma_prefetch_desc(&tmx);
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // receive buffer of the exchange, [split][W][kRecvPitch] (W: the weight
  // rows each CTA owns, fewer for the last)
  const uint32_t recv = smem_u32(smem + C::kTileBytes);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kTileBytes + C::kRecvBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kNumBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const DevErr err{args.err, args.wait_limit_ns};
  // activation rows [mb, mb + Mh) of this CTA: 65-128 rows run as two
  // 64-row halves along the grid's y (each streams the same weights; the
  // second read is an L2 hit)
  const int64_t mb = (int64_t)blockIdx.y * MP;
  const int64_t Mh = args.M - mb < MP ? args.M - mb : MP;
  const int ks = args.ksplit;  // 1..8
  const uint32_t rank = ks > 1 ? cluster_ctarank() : 0u;
  const int64_t n0 = (int64_t)(blockIdx.x / (uint32_t)ks) * 128;
  const int G = (int)(args.K / 128);
  const int kb0 = (int)((int64_t)rank * G / ks), kb1 = (int)(((int64_t)rank + 1) * G / ks);
  const int W = ((128 + ks - 1) / ks + 3) & ~3;

  auto sW = [&](int s) { return smem_u32(smem + s * C::kStageBytes); };
  auto sX = [&](int s) { return smem_u32(smem + s * C::kStageBytes + C::kWBytes); };
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[C::kStages + s]); };
  auto accf_bar = [&](int b) { return smem_u32(&bars[2 * C::kStages + b]); };
  auto acce_bar = [&](int b) { return smem_u32(&bars[2 * C::kStages + C::kAccBufs + b]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * C::kStages + 2 * C::kAccBufs]);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), C::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // the weights into L2 while the previous kernel may still run
      for (int kb = kb0; kb < kb1; ++kb) tma_prefetch_l2_2d(&tmw, kb * 128, (int32_t)n0);
      grid_dependency_wait();
      uint32_t it = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = (int)(it % C::kStages);
        const uint32_t round = it / C::kStages;
        if (!mbar_wait(empty_bar(s), (round & 1u) ^ 1u, abort_flag, err, 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(full_bar(s), C::kStageBytes);
        tma_load_2d(sW(s), &tmw, full_bar(s), kb * 128, (int32_t)n0);
        tma_load_2d(sX(s), &tmx, full_bar(s), kb * 128, (int32_t)mb);
      }
      if (!ok) {  // let the copies already in flight land before the CTA can exit
        const uint32_t first = it > (uint32_t)C::kStages ? it - C::kStages : 0u;
        for (uint32_t i = first; i < it; ++i)
          drain_wait(full_bar((int)(i % C::kStages)), (i / C::kStages) & 1u);
      }
    } else {
      grid_dependency_wait();
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    grid_dependency_wait();
    if (elect_one()) {
      // A = the weight rows (format fb), B = the activation rows (format fa)
      const uint32_t idesc = idesc_f8f6f4(128, MP, args.fb, args.fa, 0, 0);
      uint32_t it = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = (int)(it % C::kStages);
        const uint32_t buf = it & 3u, use = it >> 2;
        if (!mbar_wait(full_bar(s), (it / C::kStages) & 1u, abort_flag, err, 2) ||
            !mbar_wait(acce_bar((int)buf), (use & 1u) ^ 1u, abort_flag, err, 2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t wd = sdesc_sw128(sW(s)), xd = sdesc_sw128(sX(s));
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = 32 per MMA: 32 bytes = 2 descriptor units
          mma_f8f6f4(tmem + buf * MP, wd + 2 * k, xd + 2 * k, idesc, k != 0 ? 1u : 0u);
        mma_commit(empty_bar(s));
        mma_commit(accf_bar((int)buf));
      }
      if (!ok) {
        mma_commit(drain_bar);
        drain_wait(drain_bar, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ promotion
    grid_dependency_wait();
    const uint32_t q = warp & 3u;               // TMEM lane quadrant of this warp
    const int h = (int)(warp - 2) >> 2;         // column half (MP >= 32)
    const int64_t mcol0 = (int64_t)h * C::kCols;
    const uint32_t tbase = tmem + ((32u * q) << 16) + (uint32_t)mcol0;
    const int64_t sbo = (n0 >> 7) * G;          // this tile's weight-scale row
    float acc[C::kCols];
#pragma unroll
    for (int i = 0; i < C::kCols; ++i) acc[i] = 0.0f;
    // activation scales of columns mcol0 + 32 j + lane and the tile's weight
    // scale, loaded kQ slices ahead into register slots used round-robin
    // (a row past M gets scale 0; its accumulator column is zero anyway)
    constexpr int kQ = 4;
    uint32_t sv[kQ][C::kJ], sbq[kQ];
    auto load_s = [&](int kb, uint32_t (&v)[C::kJ], uint32_t &b) {
#pragma unroll
      for (int j = 0; j < C::kJ; ++j) {
        const int64_t m = mcol0 + 32 * j + lane;
        v[j] = m < Mh ? skinny_scale_raw<SFMT>(args.sa, (int64_t)kb * args.M + mb + m) : 0u;
      }
      b = skinny_scale_raw<SFMT>(args.sb, sbo + kb);
    };
#pragma unroll
    for (int d = 0; d < kQ; ++d)
      if (kb0 + d < kb1) load_s(kb0 + d, sv[d], sbq[d]);
    uint32_t it = 0;
    bool ok = true;
    for (int kb = kb0; kb < kb1 && ok; kb += kQ) {
#pragma unroll
      for (int jq = 0; jq < kQ; ++jq) {
        const int k = kb + jq;
        if (k >= kb1) break;
        float s[C::kJ];
        const float sbv = skinny_scale_value<SFMT>(sbq[jq]);
#pragma unroll
        for (int j = 0; j < C::kJ; ++j)
          s[j] = sv[jq][j] != 0u ? skinny_scale_value<SFMT>(sv[jq][j]) * sbv : 0.0f;
        if (k + kQ < kb1) load_s(k + kQ, sv[jq], sbq[jq]);
        const uint32_t buf = it & 3u, use = it >> 2;
        if (!mbar_wait_warp(accf_bar((int)buf), use & 1u, abort_flag, err, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r[C::kCols];
        if constexpr (C::kCols == 16) {
          FP8K_TMEM_LD_X16(tbase + buf * MP, r);
        } else {
#pragma unroll
          for (int c = 0; c < C::kCols; c += 32) FP8K_TMEM_LD_X32(tbase + buf * MP + c, (r + c));
        }
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        // the reads are complete (wait::ld): hand the buffer back at once
        if (lane == 0) mbar_arrive_relaxed(acce_bar((int)buf));
#pragma unroll
        for (int c = 0; c < C::kCols; ++c)
          acc[c] = fmaf(__shfl_sync(0xffffffffu, s[c >> 5], c & 31), __uint_as_float(r[c]), acc[c]);
        ++it;
      }
    }
    const uint32_t nl = 32 * q + lane;  // this thread's weight row in the tile
    if (ks == 1) {
      const int64_t n = n0 + nl;
      if (ok && n < args.N) {
        const float bn = args.bias != nullptr ? __ldg(args.bias + n) : 0.0f;
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(args.c) + mb * args.ldc;
#pragma unroll
        for (int c = 0; c < C::kCols; ++c) {
          const int64_t m = mcol0 + c;
          if (m < Mh) out[m * args.ldc + n] = __float2bfloat16_rn(acc[c] + bn);
        }
      }
    } else {
      // into the receive buffer of the CTA that owns this weight row, at
      // [this split][row - owner's first row][columns], 16 bytes at a time
      // and only as far as row M (after a wait gave up the values are
      // garbage; the error word says so)
      const uint32_t owner = nl / (uint32_t)W, j = nl % (uint32_t)W;
      const uint32_t dst = mapa_shared(recv, owner) +
                           ((rank * (uint32_t)W + j) * C::kRecvPitch + (uint32_t)mcol0) * 4u;
#pragma unroll
      for (int c = 0; c < C::kCols; c += 4)
        if (mcol0 + c < Mh)
          st_shared_cluster_v4(dst + (uint32_t)c * 4u, acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
    }
  }

  if (ks > 1) {
    cluster_sync();  // every partial is in its owner's receive buffer
    // this CTA's weight rows [rank W, rank W + own): the sum over the splits,
    // in split order, plus the bias, to bf16; lanes walk the owned rows
    // (consecutive output columns), warps groups of four activation rows
    const int rows = (int)Mh;
    const int own = 128 - (int)rank * W < W ? 128 - (int)rank * W : W;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(args.c) + mb * args.ldc;
    for (int m4 = (int)warp * 4; m4 < rows; m4 += C::kThreads / 32 * 4) {
      for (int j = (int)lane; j < own; j += 32) {
        const int64_t n = n0 + (int64_t)rank * W + j;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int sp = 0; sp < ks; ++sp) {
          const float4 p =
              ld_shared_f4(recv + (uint32_t)(((sp * W + j) * (int)C::kRecvPitch + m4) * 4));
          v.x += p.x; v.y += p.y; v.z += p.z; v.w += p.w;
        }
        if (n < args.N) {
          const float bn = args.bias != nullptr ? __ldg(args.bias + n) : 0.0f;
          const float r[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (m4 + i < rows) out[(int64_t)(m4 + i) * args.ldc + n] = __float2bfloat16_rn(r[i] + bn);
        }
      }
    }
    cluster_sync();  // no CTA leaves while a peer may still store into it
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// Padded activation rows per CTA for M rows (0: not a few-row shape);
// 65-128 rows take two 64-row halves.
int gemm_skinny_rows(int64_t M) {
  if (M < 1 || M > kSkinnyMaxRows) return 0;
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  return 64;
}

static int64_t skinny_halves(int64_t M) { return M > 64 ? (M + 63) / 64 : 1; }

template <int SFMT, int MP>
static cudaError_t skinny_attr(int dev) {
  static bool done[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(gemm_skinny_kernel<SFMT, MP>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SkinnyCfg<MP>::kSmem);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

// Clusters of `size` CTAs that can be resident at once (the smem opt-in is
// set first).
template <int MP>
static int skinny_active_clusters(int size) {
  using C = SkinnyCfg<MP>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || skinny_attr<0, MP>(dev) != cudaSuccess) return 0;
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
  return cudaOccupancyMaxActiveClusters(&n, gemm_skinny_kernel<0, MP>, &cfg) == cudaSuccess ? n
                                                                                          : 0;
}

static int skinny_clusters_cached(int mp, int size) {
  static int cache[64][3][kMaxClusterSplit + 1];
  static bool have[64][3][kMaxClusterSplit + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int w = mp == 16 ? 0 : mp == 32 ? 1 : 2;
  if (!have[dev][w][size]) {
    int n = 0;
    switch (w) {
      case 0: n = skinny_active_clusters<16>(size); break;
      case 1: n = skinny_active_clusters<32>(size); break;
      default: n = skinny_active_clusters<64>(size); break;
    }
    cache[dev][w][size] = n;
    have[dev][w][size] = true;
  }
  return cache[dev][w][size];
}

// K splits per 128-row weight tile: as many as the SMs hold beside the
// other tiles (one CTA per SM), at most kMaxClusterSplit and one k block
// each, and no more than let the clusters of all tiles be resident at once.
int gemm_skinny_ksplit(int64_t M, int64_t N, int64_t K, int sms) {
  const int mp = gemm_skinny_rows(M);
  if (mp == 0) return 1;
  const int64_t tiles = (N + 127) / 128 * skinny_halves(M), G = K / 128;
  int ks = kMaxClusterSplit;
  while (ks > 1 && (tiles * ks > sms || ks > G || skinny_clusters_cached(mp, ks) < tiles)) --ks;
  return ks;
}

template <int SFMT, int MP>
static cudaError_t run_skinny(const CUtensorMap &tmw, const CUtensorMap &tmx, const GemmArgs &args,
                              cudaStream_t st) {
  using C = SkinnyCfg<MP>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = skinny_attr<SFMT, MP>(dev)) != cudaSuccess) return e;
  const int ks = args.ksplit;
  if (ks < 1 || ks > kMaxClusterSplit || ks > args.K / 128)
    return cudaErrorInvalidValue;
  const int64_t tiles = (args.N + 127) / 128;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * ks), (unsigned)skinny_halves(args.M));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)ks;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ks > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<SFMT, MP>, tmw, tmx, args);
}

cudaError_t launch_gemm_skinny(int sfmt, const CUtensorMap &tmw, const CUtensorMap &tmx,
                               const GemmArgs &args, cudaStream_t st) {
  const int mp = gemm_skinny_rows(args.M);
  if (mp == 0 || args.K % 128 != 0 || args.out_dt != 1 || args.accumulate != 0)
    return cudaErrorInvalidValue;
  switch (mp) {
    case 16:
      return sfmt == 0 ? run_skinny<0, 16>(tmw, tmx, args, st) : run_skinny<1, 16>(tmw, tmx, args, st);
    case 32:
      return sfmt == 0 ? run_skinny<0, 32>(tmw, tmx, args, st) : run_skinny<1, 32>(tmw, tmx, args, st);
    default:
      return sfmt == 0 ? run_skinny<0, 64>(tmw, tmx, args, st) : run_skinny<1, 64>(tmw, tmx, args, st);
  }
}

}  // namespace fp8k
