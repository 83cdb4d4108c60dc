// Epilogue helpers shared by the GEMM kernels: output stores, split-K
// partials and the epilogue-only named barrier.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

// Store 32 consecutive results of one output row (already scaled).
__device__ __forceinline__ void store_row32(const GemmArgs &a, int64_t row, int64_t col0,
                                            const float (&v)[32]) {
  if (row >= a.M || col0 >= a.N) return;
  const bool full = (col0 + 32 <= a.N) && a.vec_store;
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

// Sum over the splits, in split order, of 32 partials of one row.
__device__ __forceinline__ void sum_partials32(const GemmArgs &a, int64_t row, int64_t col0,
                                               float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = 0.0f;
  if (row >= a.M || col0 >= a.N) return;
  const bool vec = col0 + 32 <= a.N && (a.N & 3) == 0;
  for (int sp = 0; sp < a.ksplit; ++sp) {
    const float *src = a.ws + ((int64_t)sp * a.M + row) * a.N + col0;
    if (vec) {
      const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 p = __ldcg(s4 + i);
        v[4 * i] += p.x; v[4 * i + 1] += p.y; v[4 * i + 2] += p.z; v[4 * i + 3] += p.w;
      }
    } else {
      for (int i = 0; i < 32 && col0 + i < a.N; ++i) v[i] += __ldcg(src + i);
    }
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
