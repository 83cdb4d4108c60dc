// Expert-grouped rows (MoE; Transformers fine-grained FP8, 六 6.4): the
// token rows of expert e are [offsets[e], offsets[e+1]) of A, and a kernel's
// output tiles never span two experts.  Expert e owns ceil(rows_e / tile_rows)
// * tiles_n consecutive tile indices; one warp turns the device offsets into
// that prefix (row starts and first tile indices, kept in shared memory) and
// any thread then finds a tile's expert by a binary search over it.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

// (kOn false: a one-element stand-in, so kernels without experts keep no
// table in shared memory)
template <bool kOn>
struct ExpertTiles {
  int64_t tile0[kOn ? kMaxExperts + 1 : 1];  // first tile of expert e; [E] = all tiles
  int32_t row0[kOn ? kMaxExperts + 1 : 1];   // first row of expert e; [E] = last row + 1
};

// Called by one whole warp (lane = lane_id()).  Row starts are clamped to
// [0, M], so no tile reaches past the last token even if the offsets break
// their contract (0 = offsets[0] <= ... <= offsets[E] = M).
__device__ __forceinline__ void build_expert_tiles(const int32_t *offsets, int E, int64_t M,
                                                   int64_t tiles_n, int tile_rows, uint32_t lane,
                                                   ExpertTiles<true> &x) {
  // lane l takes experts [8l, 8l + 8)
  int64_t cnt[8];
  int64_t sum = 0;
  const int32_t mm = (int32_t)M;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * (int)lane + i;
    cnt[i] = 0;
    if (e < E) {
      const int32_t r0 = min(max(offsets[e], 0), mm), r1 = min(max(offsets[e + 1], 0), mm);
      x.row0[e] = r0;
      cnt[i] = r1 > r0 ? (int64_t)((r1 - r0 + tile_rows - 1) / tile_rows) * tiles_n : 0;
      if (e == E - 1) x.row0[E] = r1;
    }
    sum += cnt[i];
  }
  int64_t incl = sum;  // inclusive scan of the lane sums
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if ((int)lane >= o) incl += v;
  }
  int64_t run = incl - sum;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = 8 * (int)lane + i;
    if (e < E) x.tile0[e] = run;
    run += cnt[i];
    if (e == E - 1) x.tile0[E] = run;
  }
}

// The expert e with tile0[e] <= t < tile0[e + 1] (empty experts skipped).
__device__ __forceinline__ int expert_of_tile(const ExpertTiles<true> &x, int E, int64_t t) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (x.tile0[mid] <= t) lo = mid; else hi = mid;
  }
  while (lo + 1 < E && x.tile0[lo + 1] <= t) ++lo;
  return lo;
}

}  // namespace fp8k
