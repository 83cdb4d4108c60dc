// Per-K-group GEMM for one activation row on the CUDA cores
// (Transformers fine-grained FP8, 一: C[m, n] = sum over 128-wide K groups g
// of sa[m, g] * sb[n / 128, g] * sum_{k in g} qa[m, k] qb[n, k]).
//
// With one row the contraction is a stream over the N x K weight codes: 2
// flop per weight byte, far below what the tensor cores need to pay off,
// and a split-K tensor-core launch spends most of its time in setup,
// pipeline fill and the cross-CTA reduction.  Here every warp owns one
// output column: its lanes stream that weight row (16-byte loads, eight in
// flight per lane), decode the codes exactly (E4M3 -> f16 -> f32), form
// 16-term dot products against the activation codes, scale each by the
// group's two factors and accumulate in fp32.  (Two to four rows measured
// no faster than the tensor-core path.)
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

constexpr int kGemvWarps = 8;   // warps (output columns) per block
constexpr int kGemvUnroll = 8;  // 16-byte weight loads in flight per lane

// Two E4M3 codes (low byte first) -> two fp32 values, exactly.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t pair) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)pair));
  return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// Dot product of two 16-code vectors in fp32.
__device__ __forceinline__ float dot16(const uint4 &x, const uint4 &y) {
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
  float d = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x0 = e4m3x2_to_float2(xw[i] & 0xFFFFu), x1 = e4m3x2_to_float2(xw[i] >> 16);
    const float2 y0 = e4m3x2_to_float2(yw[i] & 0xFFFFu), y1 = e4m3x2_to_float2(yw[i] >> 16);
    d = fmaf(x0.x, y0.x, d);
    d = fmaf(x0.y, y0.y, d);
    d = fmaf(x1.x, y1.x, d);
    d = fmaf(x1.y, y1.y, d);
  }
  return d;
}

template <int SFMT>
__device__ __forceinline__ float group_scale(const void *s, int64_t i) {
  if constexpr (SFMT == 0)
    return __ldg(static_cast<const float *>(s) + i);
  else
    return exp2_int((int)__ldg(static_cast<const uint8_t *>(s) + i) - 127);
}

// One activation row: warp w of block x owns output column kGemvWarps x + w;
// each lane takes 16-code vectors lane, lane + 32, ... of K and keeps
// kGemvUnroll of them in flight (the activation vectors are L1 hits).
template <int SFMT>
__global__ void __launch_bounds__(32 * kGemvWarps)
    gemv_group_kernel(const uint8_t *__restrict__ a, const void *__restrict__ sa,
                      const uint8_t *__restrict__ b, const void *__restrict__ sb, int64_t N,
                      int64_t K, const float *__restrict__ bias, __nv_bfloat16 *__restrict__ c) {
  const int kv = (int)(K / 16);
  const int64_t G = K / 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n = (int64_t)blockIdx.x * kGemvWarps + warp;
  if (n >= N) return;  // whole warp
  const uint4 *arow = reinterpret_cast<const uint4 *>(a);
  const uint4 *brow = reinterpret_cast<const uint4 *>(b + n * K);
  const int64_t sbn = (n >> 7) * G;
  float acc = 0.0f;
  for (int v0 = lane; v0 < kv; v0 += 32 * kGemvUnroll) {
    uint4 w[kGemvUnroll];
#pragma unroll
    for (int u = 0; u < kGemvUnroll; ++u) {
      const int v = v0 + 32 * u;
      w[u] = v < kv ? __ldcs(brow + v) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kGemvUnroll; ++u) {
      const int v = v0 + 32 * u;
      if (v >= kv) break;
      const int64_t g = v >> 3;  // eight 16-code vectors per 128-wide group
      const float s = group_scale<SFMT>(sa, g) * group_scale<SFMT>(sb, sbn + g);
      acc = fmaf(s, dot16(__ldg(arow + v), w[u]), acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) c[n] = __float2bfloat16_rn(acc + (bias != nullptr ? __ldg(bias + n) : 0.0f));
}

bool gemv_group_eligible(int64_t M, int64_t K) { return M == 1 && K % 128 == 0; }

cudaError_t launch_gemv_group(const uint8_t *a, const void *sa, const uint8_t *b, const void *sb,
                              int sfmt, int64_t M, int64_t N, int64_t K, const float *bias,
                              void *c, cudaStream_t st) {
  if (!gemv_group_eligible(M, K)) return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)((N + kGemvWarps - 1) / kGemvWarps);
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(c);
  if (sfmt == 0)
    gemv_group_kernel<0><<<blocks, 32 * kGemvWarps, 0, st>>>(a, sa, b, sb, N, K, bias, out);
  else
    gemv_group_kernel<1><<<blocks, 32 * kGemvWarps, 0, st>>>(a, sa, b, sb, N, K, bias, out);
  return cudaGetLastError();
}

}  // namespace fp8k
