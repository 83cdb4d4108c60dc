// Element-wise arithmetic of the training step that runs both in standalone
// kernels (support.cu) and inside GEMM epilogues (gemm_pair.cu): SwiGLU
// forward / backward and the AdamW update.  Every operation is an explicitly
// rounded intrinsic or a single hardware instruction (no contraction left to
// the compiler), so each value is the same wherever it is computed.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

// logistic function 1 / (1 + e^-z): the hardware exponential (__expf, a
// few fp32 ulps from e^-z) and the hardware reciprocal (rcp.approx, one
// instruction, within an fp32 ulp or so; subnormal results kept; 1 / inf =
// 0 for very negative z).  The SwiGLU values it feeds are rounded to bf16
// (8 significant bits), far coarser than either error.  (The correctly
// rounded reciprocal is a sequence of several instructions; the gated
// SwiGLU epilogue of the forward GEMM measured its arithmetic as the
// launch's limiter.)
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float sigmoidf_(float z) {
  return rcp_approx(__fadd_rn(1.0f, __expf(-z)));
}

// a = silu(h) * u = (h * s(h)) * u
__device__ __forceinline__ float swiglu_value(float h, float u) {
  return __fmul_rn(__fmul_rn(h, sigmoidf_(h)), u);
}

// dh = (da * u) * s(h) (1 + h (1 - s(h)));  du = da * (h * s(h))
__device__ __forceinline__ void swiglu_grad_values(float da, float h, float u, float &dh,
                                                   float &du) {
  const float s = sigmoidf_(h);
  const float dsilu = __fmul_rn(s, __fmaf_rn(h, __fsub_rn(1.0f, s), 1.0f));
  dh = __fmul_rn(__fmul_rn(da, u), dsilu);
  du = __fmul_rn(da, __fmul_rn(h, s));
}

// One parameter: decoupled weight decay, moment updates, bias-corrected step.
__device__ __forceinline__ void adamw1(float &p, float &m, float &v, float g, const AdamwHp &h) {
  p = __fmul_rn(p, h.decay);
  m = __fmaf_rn(h.b1, m, __fmul_rn(h.omb1, g));
  v = __fmaf_rn(h.b2, v, __fmul_rn(__fmul_rn(h.omb2, g), g));
  const float mhat = __fdiv_rn(m, h.bc1);
  const float vhat = __fdiv_rn(v, h.bc2);
  p = __fsub_rn(p, __fdiv_rn(__fmul_rn(h.lr, mhat), __fadd_rn(__fsqrt_rn(vhat), h.eps)));
}

__device__ __forceinline__ void adamw4(float4 &p, float4 &m, float4 &v, const float4 g,
                                       const AdamwHp &h) {
  adamw1(p.x, m.x, v.x, g.x, h);
  adamw1(p.y, m.y, v.y, g.y, h);
  adamw1(p.z, m.z, v.z, g.z, h);
  adamw1(p.w, m.w, v.w, g.w, h);
}

__device__ __forceinline__ uint2 f32x4_to_bf16(const float4 pv) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(pv.x, pv.y), hi = __floats2bfloat162_rn(pv.z, pv.w);
  return make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
}

// 1 - beta^t for t = the device step counter, in double, rounded to fp32.
__device__ __forceinline__ float bias_correction(double beta, int64_t t) {
  return (float)(1.0 - pow(beta, (double)t));
}

}  // namespace fp8k
