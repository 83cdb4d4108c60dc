// Per-K-group GEMM for one activation row on the CUDA cores
// (Transformers fine-grained FP8, 一: C[m, n] = sum over 128-wide K groups g
// of sa[m, g] * sb[n / 128, g] * sum_{k in g} qa[m, k] qb[n, k]).
//
// With one row the contraction is a stream over the N x K weight codes: 2
// flop per weight byte, far below what the tensor cores need to pay off,
// and a split-K tensor-core launch spends most of its time in setup,
// pipeline fill and the cross-CTA reduction.  Here a few warps share each
// output column: their lanes stream that weight row (16-byte loads, all in
// flight at once), decode the codes exactly (E4M3 -> f16 -> f32), form
// 16-term dot products against the activation codes, scale each by the
// group's two factors and accumulate in fp32.  (Two to four rows measured
// no faster than the tensor-core path.)
#include <cuda_fp16.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

constexpr int kGemvWarps = 8;   // warps per block
constexpr int kGemvSplit = 4;   // warps sharing one output column (K split)
constexpr int kGemvCols = kGemvWarps / kGemvSplit;  // output columns per block
constexpr int kGemvUnroll = 4;  // 16-byte weight loads in flight per lane

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

// One group's scale as stored (fp32, or a UE8M0 byte) and as a multiplier.
template <int SFMT>
using ScaleRaw = typename std::conditional<SFMT == 0, float, uint8_t>::type;
template <int SFMT>
__device__ __forceinline__ ScaleRaw<SFMT> load_scale(const void *s, int64_t i) {
  return __ldg(static_cast<const ScaleRaw<SFMT> *>(s) + i);
}
template <int SFMT>
__device__ __forceinline__ float scale_value(ScaleRaw<SFMT> r) {
  if constexpr (SFMT == 0)
    return r;
  else
    return exp2_int((int)r - 127);
}

// One activation row.  Block x owns output columns kGemvCols x + c; the
// kGemvSplit warps of column c take interleaved 512-byte runs of its weight
// row (warp j: 16-code vectors 32 j + lane, 32 (j + kGemvSplit) + lane, ...),
// so at K = 7168 every lane has all of its three or four weight loads in
// flight at once and the whole matrix is requested in one round trip.  The
// warps' partial sums meet in shared memory, in split order.
template <int SFMT>
__global__ void __launch_bounds__(32 * kGemvWarps)
    gemv_group_kernel(const uint8_t *__restrict__ a, const void *__restrict__ sa,
                      const uint8_t *__restrict__ b, const void *__restrict__ sb, int64_t N,
                      int64_t K, const float *__restrict__ bias, __nv_bfloat16 *__restrict__ c) {
  __shared__ float part[kGemvWarps];
  const int kv = (int)(K / 16);
  const int64_t G = K / 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = warp / kGemvSplit, split = warp % kGemvSplit;
  const int64_t n = (int64_t)blockIdx.x * kGemvCols + col;
  float acc = 0.0f;
  if (n < N) {  // whole warp
    const uint4 *arow = reinterpret_cast<const uint4 *>(a);
    const uint4 *brow = reinterpret_cast<const uint4 *>(b + n * K);
    const int64_t sbn = (n >> 7) * G;
    constexpr int kStride = 32 * kGemvSplit;
    for (int v0 = 32 * split + lane; v0 < kv; v0 += kStride * kGemvUnroll) {
      // every load of the step first (weights from HBM; activation codes and
      // scales, L2 hits), then the arithmetic: no load waits behind another
      uint4 w[kGemvUnroll], x[kGemvUnroll];
      ScaleRaw<SFMT> ra[kGemvUnroll], rb[kGemvUnroll];
#pragma unroll
      for (int u = 0; u < kGemvUnroll; ++u) {
        const int v = v0 + kStride * u;
        if (v < kv) {
          const int64_t g = v >> 3;  // eight 16-code vectors per 128-wide group
          w[u] = __ldcs(brow + v);
          x[u] = __ldg(arow + v);
          ra[u] = load_scale<SFMT>(sa, g);
          rb[u] = load_scale<SFMT>(sb, sbn + g);
        }
      }
#pragma unroll
      for (int u = 0; u < kGemvUnroll; ++u) {
        const int v = v0 + kStride * u;
        if (v >= kv) break;
        const float s = scale_value<SFMT>(ra[u]) * scale_value<SFMT>(rb[u]);
        acc = fmaf(s, dot16(x[u], w[u]), acc);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  }
  if (lane == 0) part[warp] = acc;
  __syncthreads();
  if (threadIdx.x < kGemvCols) {
    const int64_t nc = (int64_t)blockIdx.x * kGemvCols + threadIdx.x;
    if (nc < N) {
      float sum = 0.0f;
#pragma unroll
      for (int j = 0; j < kGemvSplit; ++j) sum += part[threadIdx.x * kGemvSplit + j];
      c[nc] = __float2bfloat16_rn(sum + (bias != nullptr ? __ldg(bias + nc) : 0.0f));
    }
  }
}

bool gemv_group_eligible(int64_t M, int64_t K) { return M == 1 && K % 128 == 0; }

cudaError_t launch_gemv_group(const uint8_t *a, const void *sa, const uint8_t *b, const void *sb,
                              int sfmt, int64_t M, int64_t N, int64_t K, const float *bias,
                              void *c, cudaStream_t st) {
  if (!gemv_group_eligible(M, K)) return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)((N + kGemvCols - 1) / kGemvCols);
  __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(c);
  if (sfmt == 0)
    gemv_group_kernel<0><<<blocks, 32 * kGemvWarps, 0, st>>>(a, sa, b, sb, N, K, bias, out);
  else
    gemv_group_kernel<1><<<blocks, 32 * kGemvWarps, 0, st>>>(a, sa, b, sb, N, K, bias, out);
  return cudaGetLastError();
}

}  // namespace fp8k
