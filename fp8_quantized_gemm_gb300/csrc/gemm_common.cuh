// Epilogue helpers shared by the GEMM kernels: output stores, split-K
// partials and the epilogue-only named barrier.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

// Store 32 consecutive results of one output row (already scaled), plus the
// bias of their columns when there is one.
__device__ __forceinline__ void store_row32(const GemmArgs &a, int64_t row, int64_t col0,
                                            const float (&vin)[32]) {
  if (row >= a.M || col0 >= a.N) return;
  const bool full = (col0 + 32 <= a.N) && a.vec_store;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = vin[i];
  if (a.row_scale != nullptr) {
    const float rs = __ldg(a.row_scale + row);
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i < a.N) v[i] *= rs * __ldg(a.col_scale + col0 + i);
  }
  if (a.bias != nullptr) {
    if (col0 + 32 <= a.N && (reinterpret_cast<uintptr_t>(a.bias + col0) & 15u) == 0) {
      const float4 *b4 = reinterpret_cast<const float4 *>(a.bias + col0);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 b = __ldg(b4 + i);
        v[4 * i] += b.x; v[4 * i + 1] += b.y; v[4 * i + 2] += b.z; v[4 * i + 3] += b.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (col0 + i < a.N) v[i] += __ldg(a.bias + col0 + i);
    }
  }
  if (a.out_dt == 1) {
    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.c) + row * a.ldc + col0;
    if (full) {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
      }
      uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
      for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else {
      for (int i = 0; i < 32 && col0 + i < a.N; ++i) dst[i] = __float2bfloat16_rn(v[i]);
    }
  } else {
    float *dst = static_cast<float *>(a.c) + row * a.ldc + col0;
    if (full) {
      float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float4 o = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        if (a.accumulate) {
          const float4 p = d4[i];
          o.x += p.x; o.y += p.y; o.z += p.z; o.w += p.w;
        }
        d4[i] = o;
      }
    } else {
      for (int i = 0; i < 32 && col0 + i < a.N; ++i) dst[i] = a.accumulate ? dst[i] + v[i] : v[i];
    }
  }
}

// Split-K workspace: 32 fp32 partial sums of one row for split `split`.
__device__ __forceinline__ void store_partial32(const GemmArgs &a, int split, int64_t row,
                                                int64_t col0, const float (&v)[32]) {
  if (row >= a.M || col0 >= a.N) return;
  float *dst = a.ws + ((int64_t)split * a.M + row) * a.N + col0;
  if (col0 + 32 <= a.N && (a.N & 3) == 0) {
    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i) __stcg(d4 + i, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
  } else {
    for (int i = 0; i < 32 && col0 + i < a.N; ++i) __stcg(dst + i, v[i]);
  }
}

// Store up to four consecutive results of one output row (already scaled),
// plus the bias of their columns when there is one.
__device__ __forceinline__ void store4(const GemmArgs &a, int64_t row, int64_t col, int n,
                                       const float (&vin)[4]) {
  float v[4] = {vin[0], vin[1], vin[2], vin[3]};
  if (a.row_scale != nullptr) {
    const float rs = __ldg(a.row_scale + row);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i < n) v[i] *= rs * __ldg(a.col_scale + col + i);
  }
  if (a.bias != nullptr) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i < n) v[i] += __ldg(a.bias + col + i);
  }
  if (a.out_dt == 1) {
    __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.c) + row * a.ldc + col;
    if (n == 4 && a.vec_store) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]), hi = __floats2bfloat162_rn(v[2], v[3]);
      *reinterpret_cast<uint2 *>(dst) =
          make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
    } else {
      for (int i = 0; i < n; ++i) dst[i] = __float2bfloat16_rn(v[i]);
    }
  } else {
    float *dst = static_cast<float *>(a.c) + row * a.ldc + col;
    if (n == 4 && a.vec_store) {
      float4 o = make_float4(v[0], v[1], v[2], v[3]);
      if (a.accumulate) {
        const float4 p = *reinterpret_cast<const float4 *>(dst);
        o.x += p.x; o.y += p.y; o.z += p.z; o.w += p.w;
      }
      *reinterpret_cast<float4 *>(dst) = o;
    } else {
      for (int i = 0; i < n; ++i) dst[i] = a.accumulate ? dst[i] + v[i] : v[i];
    }
  }
}

// Split K, in the CTA that arrived last for a tile: out = alpha * (sum over
// the splits, in split order, of the fp32 partials), for the whole
// tile_rows x tile_cols tile at (m0, n0).  The work is spread over all `nthr`
// epilogue threads in groups of four columns, and the partial loads of eight
// splits at a time are issued before they are added, so the reduction is
// bandwidth-bound rather than a chain of load latencies.
__device__ __forceinline__ void reduce_split_tile(const GemmArgs &a, int64_t m0, int64_t n0,
                                                  int64_t tile_rows, int64_t tile_cols,
                                                  float alpha, int tid, int nthr) {
  const int64_t rows = a.M - m0 < tile_rows ? a.M - m0 : tile_rows;
  const int64_t cols = a.N - n0 < tile_cols ? a.N - n0 : tile_cols;
  if (rows <= 0 || cols <= 0) return;
  const int64_t cg = (cols + 3) / 4;
  const bool vec = (a.N & 3) == 0;
  const int64_t plane = a.M * a.N;  // elements of one split's partials
  for (int64_t gi = tid; gi < rows * cg; gi += nthr) {
    const int64_t row = m0 + gi / cg, col = n0 + (gi % cg) * 4;
    const int n = a.N - col < 4 ? (int)(a.N - col) : 4;
    const float *src = a.ws + row * a.N + col;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (vec) {
      int sp = 0;
      for (; sp + 8 <= a.ksplit; sp += 8) {
        float4 p[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) p[u] = __ldcg(reinterpret_cast<const float4 *>(src + (sp + u) * plane));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc[0] += p[u].x; acc[1] += p[u].y; acc[2] += p[u].z; acc[3] += p[u].w;
        }
      }
      for (; sp < a.ksplit; ++sp) {
        const float4 p = __ldcg(reinterpret_cast<const float4 *>(src + sp * plane));
        acc[0] += p.x; acc[1] += p.y; acc[2] += p.z; acc[3] += p.w;
      }
    } else {
      for (int sp = 0; sp < a.ksplit; ++sp)
        for (int i = 0; i < n; ++i) acc[i] += __ldcg(src + sp * plane + i);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] *= alpha;
    store4(a, row, col, n, acc);
  }
}

// ----------------------------------------------------- split clusters --
// Row pitch (floats) of the fp32 partial tile kept in shared memory: four
// words of padding spread a warp's 32 rows over the banks.
template <int BN>
constexpr uint32_t kPartStride = BN + 4;

// 32 partials of local row `r`, columns [c, c + 32), into the partial tile.
template <int BN>
__device__ __forceinline__ void stash_partial32_bn(float *part, int r, int c, const float (&v)[32]) {
  float4 *dst = reinterpret_cast<float4 *>(part + (uint32_t)r * kPartStride<BN> + c);
#pragma unroll
  for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_shared_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// The reduction of a split cluster: CTA `rank` of the `ks` CTAs sums rows
// [rank * R / ks, (rank + 1) * R / ks) of the tile (R its valid rows) over
// every CTA's partial tile, in split order (the same order, hence the same
// sums, as the global-workspace reduction), scales by alpha and stores.
// Every thread of the CTA takes part: thread t owns float4 column t % (BN/4)
// and rows t / (BN/4), + nthr / (BN/4), ...; each step issues the remote
// loads of kStep rows of all KS splits (about 16 in flight per thread)
// before summing any, since a distributed-shared-memory load has a long
// latency.
template <int BN, int KS>
__device__ __forceinline__ void cluster_reduce_ks(const GemmArgs &a, uint32_t base, int64_t m0,
                                                  int64_t n0, int64_t r0, int64_t r1,
                                                  int64_t cols, float alpha, uint32_t rank,
                                                  int tid, int nthr) {
  constexpr int kCg = BN / 4;
  constexpr int kStep = KS >= 16 ? 1 : 16 / KS;
  const int rstride = nthr / kCg;
  if (tid >= rstride * kCg) return;
  const int64_t c = (int64_t)(tid % kCg) * 4;
  if (c >= cols) return;
  const int n = cols - c < 4 ? (int)(cols - c) : 4;
  for (int64_t rb = r0 + tid / kCg; rb < r1; rb += (int64_t)kStep * rstride) {
    float4 p[kStep][KS];
#pragma unroll
    for (int j = 0; j < kStep; ++j) {
      const int64_t r = rb + (int64_t)j * rstride;
      if (r < r1) {
        const uint32_t off = base + (uint32_t)((r * kPartStride<BN> + c) * 4);
#pragma unroll
        for (int sp = 0; sp < KS; ++sp)  // this CTA's own partial: a local load
          p[j][sp] = (uint32_t)sp == rank ? ld_shared_f4(off)
                                          : ld_shared_cluster_f4(mapa_shared(off, (uint32_t)sp));
      }
    }
#pragma unroll
    for (int j = 0; j < kStep; ++j) {
      const int64_t r = rb + (int64_t)j * rstride;
      if (r < r1) {
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int sp = 0; sp < KS; ++sp) {
          acc[0] += p[j][sp].x; acc[1] += p[j][sp].y; acc[2] += p[j][sp].z; acc[3] += p[j][sp].w;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] *= alpha;
        store4(a, m0 + r, n0 + c, n, acc);
      }
    }
  }
}

template <int BN>
__device__ __forceinline__ void cluster_reduce(const GemmArgs &a, const float *part, int64_t m0,
                                               int64_t n0, int64_t tile_rows, float alpha,
                                               uint32_t rank, int ks, int tid, int nthr) {
  const int64_t rows = a.M - m0 < tile_rows ? a.M - m0 : tile_rows;
  const int64_t cols = a.N - n0 < BN ? a.N - n0 : BN;
  if (rows <= 0 || cols <= 0) return;
  const int64_t r0 = (int64_t)rank * rows / ks, r1 = ((int64_t)rank + 1) * rows / ks;
  const uint32_t base = smem_u32(part);
  static_assert(kMaxClusterSplit == 8, "split counts below");
  switch (ks) {
    case 2: cluster_reduce_ks<BN, 2>(a, base, m0, n0, r0, r1, cols, alpha, rank, tid, nthr); break;
    case 3: cluster_reduce_ks<BN, 3>(a, base, m0, n0, r0, r1, cols, alpha, rank, tid, nthr); break;
    case 4: cluster_reduce_ks<BN, 4>(a, base, m0, n0, r0, r1, cols, alpha, rank, tid, nthr); break;
    case 5: cluster_reduce_ks<BN, 5>(a, base, m0, n0, r0, r1, cols, alpha, rank, tid, nthr); break;
    case 6: cluster_reduce_ks<BN, 6>(a, base, m0, n0, r0, r1, cols, alpha, rank, tid, nthr); break;
    case 7: cluster_reduce_ks<BN, 7>(a, base, m0, n0, r0, r1, cols, alpha, rank, tid, nthr); break;
    default: cluster_reduce_ks<BN, 8>(a, base, m0, n0, r0, r1, cols, alpha, rank, tid, nthr); break;
  }
}

// Barrier among the epilogue warps only (named barrier 1).
template <int kThreadsEpi>
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kThreadsEpi) : "memory");
}

// Barrier among the epilogue warps that returns the OR of every thread's
// predicate: one decision ("some wait ran out") for all of them before any
// further named barrier.
template <int kThreadsEpi>
__device__ __forceinline__ bool epi_any(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "r"(kThreadsEpi)
      : "memory");
  return r != 0;
}

}  // namespace fp8k
