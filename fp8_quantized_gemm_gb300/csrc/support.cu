// Elementwise support kernels of the FP8 SwiGLU training step (HBM-bound):
// SwiGLU forward / backward and the AdamW update.  16-byte vector loads,
// grid-stride loops sized to the SM count, fp32 arithmetic.
#include "common.cuh"
#include "kernels.h"
#include "support.h"

namespace fp8k {

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

__global__ void __launch_bounds__(512)
    swiglu_fwd_kernel(const uint4 *__restrict__ h, const uint4 *__restrict__ u,
                      uint4 *__restrict__ a, int64_t nvec) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    float hv[8], uv[8], av[8];
    bf16x8_to_f32(__ldcs(h + i), hv);
    bf16x8_to_f32(__ldcs(u + i), uv);
#pragma unroll
    for (int j = 0; j < 8; ++j) av[j] = hv[j] * sigmoidf_(hv[j]) * uv[j];
    __stcs(a + i, f32x8_to_bf16(av));
  }
}

__global__ void __launch_bounds__(512)
    swiglu_bwd_kernel(const uint4 *__restrict__ da, const uint4 *__restrict__ h,
                      const uint4 *__restrict__ u, uint4 *__restrict__ dh,
                      uint4 *__restrict__ du, int64_t nvec) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    float dav[8], hv[8], uv[8], dhv[8], duv[8];
    bf16x8_to_f32(__ldcs(da + i), dav);
    bf16x8_to_f32(__ldcs(h + i), hv);
    bf16x8_to_f32(__ldcs(u + i), uv);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float s = sigmoidf_(hv[j]);
      const float silu = hv[j] * s;
      dhv[j] = dav[j] * uv[j] * (s * (1.0f + hv[j] * (1.0f - s)));
      duv[j] = dav[j] * silu;
    }
    __stcs(dh + i, f32x8_to_bf16(dhv));
    __stcs(du + i, f32x8_to_bf16(duv));
  }
}

__global__ void __launch_bounds__(512)
    adamw_kernel(float4 *__restrict__ p, const float4 *__restrict__ g, float4 *__restrict__ m,
                 float4 *__restrict__ v, uint2 *__restrict__ pb, int64_t nvec, float lr,
                 float b1, float b2, float omb1, float omb2, float eps, float decay, float bc1,
                 float bc2) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    float4 pv = p[i], mv = m[i], vv = v[i];
    const float4 gv = __ldcs(g + i);
    float *pp = &pv.x, *mm = &mv.x, *vvp = &vv.x;
    const float *gg = &gv.x;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      pp[j] = pp[j] * decay;
      mm[j] = b1 * mm[j] + omb1 * gg[j];
      vvp[j] = b2 * vvp[j] + omb2 * gg[j] * gg[j];
      const float mhat = mm[j] / bc1;
      const float vhat = vvp[j] / bc2;
      pp[j] = pp[j] - lr * mhat / (sqrtf(vhat) + eps);
    }
    p[i] = pv;
    m[i] = mv;
    v[i] = vv;
    if (pb != nullptr) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(pv.x, pv.y), hi = __floats2bfloat162_rn(pv.z, pv.w);
      pb[i] = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
    }
  }
}

static int blocks_for(int64_t nvec, int threads, int sms) {
  const int64_t need = (nvec + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 4;
  return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

cudaError_t launch_swiglu_fwd(const void *h, const void *u, void *a, int64_t n, int sms,
                              cudaStream_t st) {
  const int64_t nvec = n / 8;
  swiglu_fwd_kernel<<<blocks_for(nvec, 512, sms), 512, 0, st>>>(
      static_cast<const uint4 *>(h), static_cast<const uint4 *>(u), static_cast<uint4 *>(a), nvec);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(const void *da, const void *h, const void *u, void *dh, void *du,
                              int64_t n, int sms, cudaStream_t st) {
  const int64_t nvec = n / 8;
  swiglu_bwd_kernel<<<blocks_for(nvec, 512, sms), 512, 0, st>>>(
      static_cast<const uint4 *>(da), static_cast<const uint4 *>(h), static_cast<const uint4 *>(u),
      static_cast<uint4 *>(dh), static_cast<uint4 *>(du), nvec);
  return cudaGetLastError();
}

cudaError_t launch_adamw(float *p, const float *g, float *m, float *v, void *pb, int64_t n,
                         int64_t step, double lr, double b1, double b2, double eps, double wd, int sms,
                         cudaStream_t st) {
  const int64_t nvec = n / 4;
  // 1 - beta and the bias corrections are formed in double on the host: in
  // fp32, 1 - 0.999f is off by 1.3e-5 relative
  const float bc1 = (float)(1.0 - pow(b1, (double)step));
  const float bc2 = (float)(1.0 - pow(b2, (double)step));
  const float omb1 = (float)(1.0 - b1), omb2 = (float)(1.0 - b2);
  adamw_kernel<<<blocks_for(nvec, 512, sms), 512, 0, st>>>(
      reinterpret_cast<float4 *>(p), reinterpret_cast<const float4 *>(g),
      reinterpret_cast<float4 *>(m), reinterpret_cast<float4 *>(v), static_cast<uint2 *>(pb), nvec,
      (float)lr, (float)b1, (float)b2, omb1, omb2, (float)eps, (float)(1.0 - lr * wd), bc1, bc2);
  return cudaGetLastError();
}

}  // namespace fp8k
