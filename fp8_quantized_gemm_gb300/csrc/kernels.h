// Host-side launch entry points of the device kernels (internal to the
// library; the public C ABI is include/fp8gemm.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8k {

// fp32 hyperparameters of one AdamW update: 1 - beta and the decay factor
// 1 - lr * wd formed in double on the host; the bias corrections 1 - beta^t
// (bc1, bc2) in double on the device from the step counter.
struct AdamwHp {
  float lr, b1, b2, omb1, omb2, eps, decay, bc1, bc2;
};

cudaError_t launch_amax(const void *x, int in_dt, int64_t n, float *out, int sms,
                        cudaStream_t st);
cudaError_t launch_quant_tensor(const void *x, int in_dt, int64_t rows, int64_t cols, int fmt,
                                const float *amax_in, const float *scale, float *scale_out,
                                uint8_t *q, uint8_t *qt, float *amax_out, int sms,
                                cudaStream_t st);
cudaError_t launch_quant_group(const void *x, int in_dt, int64_t M, int64_t K, int fmt,
                               int sfmt, uint8_t *q, void *scales, int sms, cudaStream_t st);
cudaError_t launch_quant_block(const void *w, int in_dt, int64_t N, int64_t K, int fmt,
                               int sfmt, uint8_t *q, void *scales, cudaStream_t st);
// amax == nullptr: one-level MXFP8; per_row: amax and global_out are [R]
cudaError_t launch_quant_mx(const void *x, int in_dt, int64_t R, int64_t K, int fmt,
                            const float *amax, float *global_out, uint8_t *q, uint32_t *local,
                            int sms, cudaStream_t st, bool per_row = false);
cudaError_t launch_row_amax(const void *x, int in_dt, int64_t R, int64_t K, float *out, int sms,
                            cudaStream_t st);
// Per-K-group GEMM of one activation row on the CUDA cores (gemv.cu): bf16
// output [1, N], optional fp32 bias; K % 128 == 0.
bool gemv_group_eligible(int64_t M, int64_t K);
cudaError_t launch_gemv_group(const uint8_t *a, const void *sa, const uint8_t *b, const void *sb,
                              int sfmt, int64_t M, int64_t N, int64_t K, const float *bias,
                              void *c, cudaStream_t st);
cudaError_t launch_ue8m0_words(const uint8_t *sa, const uint8_t *sb, int64_t M, int64_t N,
                               int64_t K, uint32_t *la, uint32_t *lb, int sms, cudaStream_t st);
cudaError_t launch_ue8m0_words_experts(const uint8_t *sa, const uint8_t *sb,
                                       const int32_t *offsets, int E, int64_t M, int64_t N,
                                       int64_t K, int64_t tmax, uint32_t *la, uint32_t *lb,
                                       int sms, cudaStream_t st);
cudaError_t launch_quant_block32(const void *w, int in_dt, int64_t N, int64_t K, int fmt,
                                 uint8_t *q, uint8_t *scales, uint32_t *local, int sms,
                                 cudaStream_t st);
// (32, 32) weight blocks with fp32 scales [ceil(N/32), K/32] (no MX words).
cudaError_t launch_quant_block32_f32(const void *w, int in_dt, int64_t N, int64_t K, int fmt,
                                     uint8_t *q, float *scales, int sms, cudaStream_t st);
// 1 x 32 token groups (scales group-major [ceil(K/32), M], fp32 or UE8M0).
cudaError_t launch_quant_group32(const void *x, int in_dt, int64_t M, int64_t K, int fmt,
                                 int sfmt, uint8_t *q, void *scales, int sms, cudaStream_t st);
cudaError_t launch_dequant_block(const uint8_t *q, int64_t N, int64_t K, int fmt, int sfmt,
                                 const void *scales, void *out, int sms, cudaStream_t st);
cudaError_t launch_auto_scale(const float *amax0, double grow, int fmt, float *scale,
                              cudaStream_t st);
cudaError_t launch_delayed_update(float *hist, float *scale, const float *amax_cur, int64_t L,
                                  int fmt, cudaStream_t st);
// Up to kMaxDelayed amax-history steps in one launch (one CTA each).
constexpr int kMaxDelayed = 16;
struct DelayedItems {
  float *hist[kMaxDelayed];
  float *scale[kMaxDelayed];
  const float *amax_cur[kMaxDelayed];
  int64_t L[kMaxDelayed];
  int fmt[kMaxDelayed];
  int count;
};
cudaError_t launch_delayed_update_multi(const DelayedItems &items, cudaStream_t st);

// Current scaling of up to kMaxMulti tensors in one cooperative launch
// (quantize_multi.cu).  `sync` is device scratch of 2 * kMaxMulti uint32
// words (keys, then arrival counters), cleared by the launcher.
constexpr int kMaxMulti = 4;
struct MultiQuantArgs {
  const void *x[kMaxMulti];
  int64_t n[kMaxMulti];
  int fmt[kMaxMulti];
  uint8_t *q[kMaxMulti];
  float *amax_out[kMaxMulti];   // nullable
  float *scale_out[kMaxMulti];
  int count;
  uint32_t *sync;
  uint32_t *err;               // device error word
  uint64_t wait_limit_ns;      // bound of every wait
};
cudaError_t launch_quant_multi(const MultiQuantArgs &args, int in_dt, int sms, cudaStream_t st);

// GEMM family.  Scale modes of the epilogue / main loop:
enum GemmScaleMode : int {
  kScaleTensor = 0,      // per-tensor: alpha = sa[0] * sb[0] in the epilogue
  kScaleMx = 1,          // block-scaled MMA, packed E8M0 words; alpha = ga[0] * gb[0] (1 if ga null)
  kScaleGroupUe8m0 = 2,  // block-scaled MMA, per-128 UE8M0 bytes replicated in-kernel
  kScaleGroupF32 = 3,    // per-128 fp32 scales promoted on the CUDA cores
  kScaleGroupF32x32 = 4  // fp32 scales per 1x32 activation group and 32x32 weight
                         // block: every K=32 MMA into its own TMEM buffer, promoted
};

struct GemmArgs {
  int64_t M, N, K;
  int fa, fb;          // operand formats: 0 = E4M3, 1 = E5M2
  int out_dt;          // 0 = f32, 1 = bf16
  int accumulate;      // f32 output only
  int vec_store;       // 1: c and ldc allow 16-byte vector stores
  int a_mn, b_mn;      // 1: operand stored MN-major ([K, M] / [K, N]); per-tensor mode only
  int64_t ldc;
  void *c;
  const void *sa, *sb;         // scale operands (meaning depends on the mode)
  const float *ga, *gb;        // global factors (kScaleMx)
  uint32_t *err;               // device error word
  uint64_t wait_limit_ns;      // bound of every mbarrier wait
  // split-K (small M): ksplit > 1 splits every tile's K range; fp32 partials
  // go to ws [ksplit][M][N] and counters[tile] counts finished splits (the
  // last one reduces in split order and resets the counter to 0)
  int ksplit;
  float *ws;
  uint32_t *counters;
  // cluster_split: the ksplit CTAs of a tile form one thread-block cluster
  // (cluster rank = split) and reduce their partials through distributed
  // shared memory; ws and counters are then unused
  int cluster_split;
  // experts > 0 (group modes, ksplit 1): rows [offsets[e], offsets[e+1]) of A
  // use expert e's weights: B rows e*N .. e*N+N-1 of the [E*N, K] tensor map
  // and scales sb + e * sb_expert_stride
  int experts;
  const int32_t *offsets;       // device, experts + 1 entries
  int64_t sb_expert_stride;     // elements of sb per expert
  // nullable fp32 [N]: added to every row of the result (after the scales,
  // before the output cast)
  const float *bias;
  // nullable fp32 [M] and [N] (together): the result is multiplied by
  // row_scale[m] * col_scale[n] (per-row global factors of two-level scaling)
  const float *row_scale, *col_scale;
  // 1 (block-scaled and FP32-promotion modes, ksplit 1, K-major B, no
  // experts): clusters of two CTAs on vertically adjacent tiles multicast
  // the B boxes (the B tensor map's box is then BN / 2 rows)
  int multicast;
  // 1 (CTA-pair kernel; no accumulate, 16-byte aligned c and pitch): the
  // epilogue writes C through shared memory with TMA stores of 32-row x
  // 128-byte boxes (the kernel gets the output tensor map separately)
  int tma_store;
  // AdamW epilogue (CTA-pair kernel): the fp32 result sa*sb*A*B^T is the
  // gradient of the parameters adam_p [M, ldc] (moments adam_m, adam_v, bf16
  // copy adam_pb, nullable), which it updates in place at step t =
  // *adam_step; c is not written
  float *adam_p, *adam_m, *adam_v;
  void *adam_pb;
  const int64_t *adam_step;
  AdamwHp adam_hp;  // bc1, bc2 formed in the kernel
  double adam_b1d, adam_b2d;
  // Gated SwiGLU epilogue (CTA-pair kernel): in each pair, rank 0 stages
  // rows of B and rank 1 the same rows of a second weight (its own tensor
  // map; dequant scale swi_sb2), so one 256 x 256 accumulator holds h
  // (columns 0-127) and u (128-255) of the same 128 output columns.  The
  // epilogue writes c <- bf16(h), swi_u <- bf16(u) and swi_q <- the codes of
  // a = bf16(silu(h) u) divided by *swi_scale (format swi_fmt), all [M, ldc],
  // and folds max |a| into *swi_amax (cleared by the launcher)
  int gated;
  const float *swi_sb2;
  void *swi_u;
  uint8_t *swi_q;
  const float *swi_scale;
  uint32_t *swi_amax;
  int swi_fmt;
};
constexpr int kMaxExperts = 256;

// Wait bound the API passes to kernels (fp8_set_option FP8_OPT_WAIT_LIMIT_NS).
uint64_t wait_limit_ns();

// Split count the launcher would use for this shape (1 = no split);
// `cluster`: the splits reduce through a cluster (at most kMaxClusterSplit,
// no partials in global memory) rather than through a global workspace.
constexpr int kMaxClusterSplit = 8;
int gemm_ksplit(int mode, int64_t M, int64_t N, int64_t K, int sms, bool cluster);

// Output-tile width (N) of a mode at M rows; the B tensor map's box uses it.
int gemm_tile_n(int mode, int64_t M, int64_t N, int sms);

// Per-K-group GEMM for 1 <= M <= kSkinnyMaxRows activation rows
// (gemm_skinny.cu; beyond 64 rows, 64-row halves along the grid's y): bf16
// output, optional bias, K % 128 == 0.  tmw: the weights [N, K] with
// 128 x 128 boxes; tmx: the activations [M, K] with boxes of
// gemm_skinny_rows(M) rows x 128.  args.ksplit = gemm_skinny_ksplit(...).
constexpr int64_t kSkinnyMaxRows = 128;
int gemm_skinny_rows(int64_t M);
int gemm_skinny_ksplit(int64_t M, int64_t N, int64_t K, int sms);
cudaError_t launch_gemm_skinny(int sfmt, const CUtensorMap &tmw, const CUtensorMap &tmx,
                               const GemmArgs &args, cudaStream_t st);

cudaError_t launch_gemm(int mode, const CUtensorMap &tma, const CUtensorMap &tmb,
                        const GemmArgs &args, int sms, cudaStream_t st);
// Expert-grouped per-K-group GEMM (args.experts > 0) with B tiles `bn` wide.
cudaError_t launch_gemm_experts(int mode, int bn, const CUtensorMap &tma, const CUtensorMap &tmb,
                                const GemmArgs &args, int sms, cudaStream_t st);

// CTA-pair (cta_group::2) variant of the per-tensor GEMM: 256 x 256 tiles, B
// staged half per CTA (the B tensor map box has gemm_pair_b_rows() rows).
bool gemm_pair_eligible(int mode, int64_t M, int64_t N, int sms);
constexpr int kMaxGroup = 4;  // problems per grouped launch
// One launch over `count` independent per-tensor problems (longest K first).
// tmc[i]: the output tensor map of problem i (read when args[i].tma_store).
// tmb2[i]: the second weight of a gated problem (read when args[i].gated;
// tmb2 may be null when no problem is gated).
cudaError_t launch_gemm_pair_group(const CUtensorMap *tma, const CUtensorMap *tmb,
                                   const CUtensorMap *tmc, const CUtensorMap *tmb2,
                                   const GemmArgs *args, int count, int sms, cudaStream_t st);
int gemm_pair_b_rows();
// 256-row tiles per band of the CTA-pair tile order (fp8_set_option).
int64_t gemm_pair_band_rows();
cudaError_t launch_gemm_pair(const CUtensorMap &tma, const CUtensorMap &tmb,
                             const CUtensorMap &tmc, const GemmArgs &args, int sms,
                             cudaStream_t st);

// CTA-pair variant of the FP32-scale per-group GEMM (kScaleGroupF32):
// 256 x 256 tiles, the per-slice promotion in both CTAs' epilogues; K-major
// operands, K % 128 == 0, no split K; plain or expert-grouped rows
// (args.experts, args.offsets, args.sb_expert_stride as for
// launch_gemm_experts, B's tensor map over all experts' rows).  The B tensor
// map box has gemm_pair_promote_b_rows() rows.
bool gemm_pair_promote_eligible(int64_t M, int64_t N, int64_t K, int sms);
int gemm_pair_promote_b_rows();
cudaError_t launch_gemm_pair_promote(const CUtensorMap &tma, const CUtensorMap &tmb,
                                     const GemmArgs &args, int sms, cudaStream_t st);

}  // namespace fp8k
