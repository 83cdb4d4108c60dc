// Launchers of the elementwise support kernels (SwiGLU, AdamW).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "elementwise.cuh"

namespace fp8k {

cudaError_t launch_swiglu_fwd(const void *h, const void *u, void *a, int64_t n, int sms,
                              cudaStream_t st);
cudaError_t launch_swiglu_bwd(const void *da, const void *h, const void *u, void *dh, void *du,
                              int64_t n, int sms, cudaStream_t st);
// SwiGLU fused with delayed-scaling quantization of its output(s): codes of
// the bf16 result divided by the given scale, fused amax (nullable; clears it
// first).
cudaError_t launch_swiglu_fwd_quant(const void *h, const void *u, int64_t n, int fmt,
                                    const float *scale, uint8_t *q, float *amax_out, int sms,
                                    cudaStream_t st);
cudaError_t launch_swiglu_bwd_quant(const void *da, const void *h, const void *u, int64_t n,
                                    int fmt, const float *scale_h, const float *scale_u,
                                    uint8_t *qh, uint8_t *qu, float *amax_h, float *amax_u,
                                    int sms, cudaStream_t st);
cudaError_t launch_adamw(float *p, const float *g, float *m, float *v, void *pb, int64_t n,
                         int64_t step, double lr, double b1, double b2, double eps, double wd, int sms,
                         cudaStream_t st);

// Multi-tensor AdamW with the step counter on the device.
constexpr int kMaxAdamw = 8;
struct AdamwMulti {
  float *p[kMaxAdamw];
  const float *g[kMaxAdamw];
  float *m[kMaxAdamw];
  float *v[kMaxAdamw];
  void *pb[kMaxAdamw];  // nullable bf16 copies
  int64_t n[kMaxAdamw];
  // nullable: codes of bf16(p) under q_scale[0] (format q_fmt) and their
  // amax (nullable; cleared by the launcher), the next step's quantization
  uint8_t *q[kMaxAdamw];
  const float *q_scale[kMaxAdamw];
  uint32_t *q_amax[kMaxAdamw];
  int q_fmt[kMaxAdamw];
  int count;
  int64_t *step;        // device: read as t (incremented first when advancing)
  AdamwHp hp;           // set by the launcher (bias corrections: in the kernel)
  double b1d, b2d;
};
// The fp32 hyperparameters of an AdamW update (1 - beta, decay in double).
AdamwHp adamw_hp(double lr, double b1, double b2, double eps, double wd);
cudaError_t launch_adamw_multi(AdamwMulti a, bool advance, double lr, double b1, double b2,
                               double eps, double wd, int sms, cudaStream_t st);

}  // namespace fp8k
