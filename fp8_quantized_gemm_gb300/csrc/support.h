// Launchers of the elementwise support kernels (SwiGLU, AdamW).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8k {

cudaError_t launch_swiglu_fwd(const void *h, const void *u, void *a, int64_t n, int sms,
                              cudaStream_t st);
cudaError_t launch_swiglu_bwd(const void *da, const void *h, const void *u, void *dh, void *du,
                              int64_t n, int sms, cudaStream_t st);
cudaError_t launch_adamw(float *p, const float *g, float *m, float *v, void *pb, int64_t n,
                         int64_t step, double lr, double b1, double b2, double eps, double wd, int sms,
                         cudaStream_t st);

}  // namespace fp8k
