// Element-wise arithmetic of the training step that runs both in standalone
// kernels (support.cu) and inside GEMM epilogues (gemm_pair.cu): SwiGLU
// forward / backward and the AdamW update.  Every operation is an explicitly
// rounded intrinsic or a single hardware instruction (no contraction left to
// the compiler), so each value is the same wherever it is computed.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace fp8k {

// e^-z as 2^(-z log2 e): the product rounded once, then the hardware
// base-2 exponential (ex2.approx.ftz, relative error near 2^-22).  Its
// flush of subnormals changes no logistic value: a subnormal argument gives
// 1 either way, and a subnormal result (z > 87) vanishes in 1 + e^-z.
__device__ __forceinline__ float ex2_approx_ftz(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}
constexpr float kNegLog2e = -1.4426950408889634f;

// logistic function 1 / (1 + e^-z): the exponential above and the hardware
// reciprocal (rcp.approx, one instruction, within an fp32 ulp or so;
// subnormal results kept; 1 / inf = 0 for very negative z).  The SwiGLU
// values it feeds are rounded to bf16 (8 significant bits), far coarser
// than either error.  (The correctly rounded reciprocal is a sequence of
// several instructions; the gated SwiGLU epilogue of the forward GEMM
// measured its arithmetic as the launch's limiter.)
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float sigmoidf_(float z) {
  return rcp_approx(__fadd_rn(1.0f, ex2_approx_ftz(__fmul_rn(z, kNegLog2e))));
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

// The same two values at a time: every product, sum and fma above issued as
// one packed f32x2 instruction (each half rounded as the scalar instruction;
// 1 - s as fma(s, -1, 1), the same single rounding), the exponential and
// the reciprocal per value.  Bit-identical to the scalar forms.
__device__ __forceinline__ uint64_t sigmoid2(uint64_t H) {
  float t0, t1, p0, p1;
  f32x2_unpack(f32x2_mul(H, f32x2_pack(kNegLog2e, kNegLog2e)), t0, t1);
  f32x2_unpack(f32x2_add(f32x2_pack(ex2_approx_ftz(t0), ex2_approx_ftz(t1)),
                         f32x2_pack(1.0f, 1.0f)),
               p0, p1);
  return f32x2_pack(rcp_approx(p0), rcp_approx(p1));
}

__device__ __forceinline__ void swiglu_value2(float h0, float h1, float u0, float u1, float &a0,
                                              float &a1) {
  const uint64_t H = f32x2_pack(h0, h1);
  f32x2_unpack(f32x2_mul(f32x2_mul(H, sigmoid2(H)), f32x2_pack(u0, u1)), a0, a1);
}

__device__ __forceinline__ void swiglu_grad8(const float (&da)[8], const float (&h)[8],
                                             const float (&u)[8], float (&dh)[8],
                                             float (&du)[8]) {
  const uint64_t one = f32x2_pack(1.0f, 1.0f), mone = f32x2_pack(-1.0f, -1.0f);
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    const uint64_t H = f32x2_pack(h[j], h[j + 1]), U = f32x2_pack(u[j], u[j + 1]),
                   D = f32x2_pack(da[j], da[j + 1]);
    const uint64_t S = sigmoid2(H);
    const uint64_t dsilu = f32x2_mul(S, f32x2_fma(H, f32x2_fma(S, mone, one), one));
    f32x2_unpack(f32x2_mul(f32x2_mul(D, U), dsilu), dh[j], dh[j + 1]);
    f32x2_unpack(f32x2_mul(D, f32x2_mul(H, S)), du[j], du[j + 1]);
  }
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
