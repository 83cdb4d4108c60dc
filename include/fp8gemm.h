/*
 * fp8gemm.h -- C ABI of the scaled-FP8 GEMM library (libfp8gemm.so), sm_103a.
 *
 * The library quantizes operands to E4M3 / E5M2 and contracts them on the
 * tcgen05 tensor cores with FP32 accumulation, applying the scales in one of
 * four places: per tensor in the epilogue (current or delayed scaling), per
 * K group in the main loop (1x128 x 128x128, FP32 or UE8M0 scales), or two
 * level (E8M0 local factors inside block-scaled MMA, an FP32 global factor in
 * the epilogue).
 *
 * Sources (web pages, by title and section):
 *   [Flax]   "Flax FP8 量化实战指南" -- 1 (Q/DQ), 2.2 (current scaling,
 *            quantize/dequantize), 2.3 (delayed scaling, amax history),
 *            3.3 (E4M3 forward / E5M2 gradients), 5.1 (meta state).
 *   [Nano]   "Nanochat的FP8训练模块" -- "核心原语" (_scaled_mm, TN layout),
 *            "实现" (forward / backward GEMMs, E5M2 max 57344).
 *   [HF]     "Transformers 中的细粒度 FP8 量化配置..." -- 一 (128x128 weight
 *            blocks, 1x128 token groups, weight_scale_inv shape), 四
 *            (scale_fmt float | ue8m0), 七 (UE8M0 rounded up, quantize with it).
 *   [MOSS]   "MOSS: 高效、精确的 FP8 LLM 训练" -- 4 (two-level microscaling,
 *            steps 1-4).
 *
 * Conventions shared by every call
 * --------------------------------
 * - All data pointers are DEVICE pointers on the current CUDA device; the
 *   caller owns every buffer (allocates and frees it).  The library never
 *   frees or retains a caller pointer past the call.
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *   default stream).  A return of FP8_OK means the work was enqueued.
 * - A "scale" is always the DEQUANT multiplier amax / MAX ([Flax] 1, 2.2):
 *   quantize divides by it, dequantize multiplies by it.
 * - Matrices are row-major.  GEMM operands are both stored [rows, K] with K
 *   contiguous ("A row-major, B column-major", the TN layout of [Nano]
 *   "核心原语"); b is [N, K], the layout of nn.Linear.weight.
 * - Quantization is bit-exact: y = fl32(x / s) (IEEE division), clipped to
 *   +-MAX, then one round-to-nearest-even cast ([Flax] 2.2 quantize).
 * - Errors: calls return an fp8_status_t.  Device-side errors (a bounded wait
 *   that expired) are recorded in a library-wide device error word and read
 *   with fp8_get_last_device_error().
 */
#ifndef FP8GEMM_H
#define FP8GEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8_API __attribute__((visibility("default")))
#else
#define FP8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *fp8_stream_t; /* == cudaStream_t */

typedef enum {
  FP8_OK = 0,
  FP8_ERR_INVALID_ARG = -1, /* null pointer, non-positive or too-large size, bad enum */
  FP8_ERR_MISALIGNED = -2,  /* pointer/stride alignment or K granularity violated */
  FP8_ERR_UNSUPPORTED = -3, /* format combination or shape the kernels do not cover */
  FP8_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed */
  FP8_ERR_TIMEOUT = -5,     /* a device-side bounded wait expired (device error word) */
  FP8_ERR_NO_DEVICE = -6,   /* no sm_103 device is current */
  FP8_ERR_SCRATCH_LIMIT = -7 /* shape needs more than fp8_gemm_group_noalloc's fixed scratch */
} fp8_status_t;

typedef enum { FP8_IN_BF16 = 0, FP8_IN_F32 = 1 } fp8_in_dtype_t;
typedef enum { FP8_E4M3 = 0, FP8_E5M2 = 1 } fp8_fmt_t; /* E4M3fn max 448, E5M2 max 57344 */
typedef enum { FP8_SCALE_F32 = 0, FP8_SCALE_UE8M0 = 1 } fp8_scale_fmt_t;
typedef enum { FP8_OUT_F32 = 0, FP8_OUT_BF16 = 1 } fp8_out_dtype_t;
/* Storage of a GEMM operand of logical shape [R, K] (R = M for A, N for B):
 * K-major = [R, K] row-major (K contiguous); MN-major = [K, R] row-major (R
 * contiguous), i.e. the row-major codes of the transposed operand. */
typedef enum { FP8_K_MAJOR = 0, FP8_MN_MAJOR = 1 } fp8_layout_t;

/* ------------------------------------------------------------------ amax --
 * fp8_amax: amax_out[0] = max |x[i]| over i < n ([Flax] 1: "amax is the max
 * absolute value of the tensor").  x: n elements of in_dt, 16-byte aligned.
 * amax_out: one fp32, overwritten (the call clears it first).  Exact (max is
 * order independent).  n == 0 gives 0.
 */
FP8_API int fp8_amax(const void *x, int in_dt, int64_t n, float *amax_out, fp8_stream_t stream);

/* ------------------------------------------------------- quantize tensor --
 * fp8_quantize_tensor: per-tensor quantization ([Flax] 2.2 quantize; 2.3
 * in_q for delayed scaling).
 *   x       [rows, cols] of in_dt, row-major, 16-byte aligned, cols % 8 == 0.
 *   fmt     FP8_E4M3 (activations, weights) or FP8_E5M2 (gradients).
 *   amax_in nullable.  CURRENT scaling: when non-null the scale is
 *           s = fl32(amax_in[0] / MAX) (1.0 if amax_in[0] == 0), typically the
 *           output of fp8_amax on the same x.
 *   scale   DELAYED scaling: used when amax_in is null; s = scale[0] (the
 *           scale fp8_delayed_state_update left for this step).
 *   scale_out nullable; receives s (fp32), e.g. for the GEMM epilogue.
 *   q       [rows, cols] uint8 codes, row-major.
 *   q_t     nullable; [cols, rows] uint8 codes: the transposed copy that the
 *           backward GEMMs read as a K-contiguous operand.
 *   amax_out nullable; receives max |x| (cleared first), the amax that the
 *           delayed-scaling history takes for this step.  Must not alias
 *           amax_in or scale (INVALID_ARG).
 *   Codes: q = RNE_fp8(clip(fl32(x / s), -MAX, MAX)) for finite x; +-inf
 *   gives +-MAX; a NaN x gives a NaN code (its sign bit may follow x's).
 */
FP8_API int fp8_quantize_tensor(const void *x, int in_dt, int64_t rows, int64_t cols, int fmt,
                        const float *amax_in, const float *scale, float *scale_out,
                        uint8_t *q, uint8_t *q_t, float *amax_out, fp8_stream_t stream);

/* ------------------------------------------ quantize, several tensors --
 * fp8_quantize_tensors: current scaling ([Flax] 2.2) of `count` (1..4)
 * tensors in ONE launch.  For each item: amax = max |x|, scale =
 * fl32(amax / MAX) (1.0 for amax 0), q = RNE_fp8(clip(x / scale)) -- the same
 * amax, scale and bytes as fp8_amax followed by fp8_quantize_tensor with
 * amax_in.  Row-major codes only (the per-tensor GEMMs read them K- or
 * MN-major).  The items are pipelined: while one tensor is divided and
 * cast, the next is being reduced; the smallest item goes first (its amax
 * pass runs alone), the others follow in the order given.  The order changes
 * no result.
 *   items  HOST array of `count` descriptors (read during the call only).
 *     x         device, 16-byte aligned, n >= 0 elements of in_dt (every item
 *               the same in_dt, else FP8_ERR_UNSUPPORTED)
 *     q         device, 16-byte aligned, n bytes; must not overlap any x
 *               (x and q may be null when n == 0: the item then reports
 *               amax 0 and scale 1.0)
 *     amax_out  nullable device fp32;  scale_out  device fp32 (required,
 *               distinct from amax_out)
 *   sync   device scratch of FP8_QUANT_SYNC_WORDS uint32 words, 16-byte
 *          aligned, owned by the caller: the call clears it (a memset on
 *          `stream`) and the kernel's CTAs count themselves in there.  Calls
 *          that can run at the same time need distinct scratch.  Nothing is
 *          allocated, so the call can be captured into a CUDA graph.
 * Runs as a cooperative launch (one CTA per SM, all resident at once: its
 * quantize warps wait for every CTA's share of the amax, bounded by the wait
 * limit; FP8_ERR_TIMEOUT is then reported by fp8_get_last_device_error).
 */
#define FP8_QUANT_SYNC_WORDS 8
typedef struct {
  const void *x;
  int in_dt;
  int64_t n;
  int fmt;
  uint8_t *q;
  float *amax_out;
  float *scale_out;
} fp8_quant_item_t;

FP8_API int fp8_quantize_tensors(const fp8_quant_item_t *items, int count, uint32_t *sync,
                                 fp8_stream_t stream);

/* -------------------------------------------------- quantize token group --
 * fp8_quantize_token_group: dynamic per-token activation quantization in
 * 1 x 128 K groups ([HF] 一; scale formats [HF] 四/七).
 *   x      [M, K] of in_dt, row-major, 16-byte aligned, K % 16 == 0 (the last
 *          group may be ragged: its amax covers the valid elements only).
 *   sfmt   FP8_SCALE_F32: scales are fp32 amax/MAX (1.0 for an all-zero group).
 *          FP8_SCALE_UE8M0: scales are bytes e + 127 with 2^e = amax/MAX
 *          rounded UP to a power of two (byte 127 for an all-zero group), and
 *          the group is quantized WITH 2^e ([HF] 七).
 *   q      [M, K] uint8 codes.
 *   scales GROUP-MAJOR: [ceil(K/128), M] (fp32 or uint8): scales[g * M + m] is
 *          the scale of row m, K group g.
 */
FP8_API int fp8_quantize_token_group(const void *x, int in_dt, int64_t M, int64_t K, int fmt,
                             int sfmt, uint8_t *q, void *scales, fp8_stream_t stream);

/* -------------------------------------------------------- quantize block --
 * fp8_quantize_block: 128 x 128 weight-block quantization ([HF] 一: one scale
 * per block, weight_scale_inv of shape (ceil(N/128), ceil(K/128))).
 *   w      [N, K] of in_dt, row-major, 16-byte aligned, K % 16 == 0.
 *   sfmt   as for fp8_quantize_token_group.
 *   q      [N, K] uint8 codes.
 *   scales [ceil(N/128), ceil(K/128)] row-major (fp32 or uint8).
 */
FP8_API int fp8_quantize_block(const void *w, int in_dt, int64_t N, int64_t K, int fmt, int sfmt,
                       uint8_t *q, void *scales, fp8_stream_t stream);

/* ----------------------------------------------------------- quantize mx --
 * fp8_quantize_mx: MOSS two-level microscaling ([MOSS] 4, steps 1-4).
 *   x      [R, K] of in_dt, row-major, 16-byte aligned, K % 128 == 0.
 *   amax   device fp32: max |x| over the whole tensor (from fp8_amax).  The
 *          global factor is S = max_i s_i with s_i = fl32(amax_i / MAX) over
 *          the 1x32 blocks; since fp32 rounding is monotone this equals
 *          fl32(amax / MAX), which is how it is evaluated (1.0 if amax == 0).
 *   global_out device fp32: receives S (the FP32 factor the GEMM epilogue
 *          applies).
 *   q      [R, K] uint8 codes, quantized with the effective scale S * r_i.
 *   local  E8M0 local factors r_i = 2^ceil(log2(fl32(s_i / S))) in (0, 1],
 *          byte e + 127 (byte 127 for an all-zero block; e clamped at -127).
 *          Layout (the block-scaled GEMM's operand layout): R_pad = R rounded
 *          up to 128; local is uint32 [K/128][R_pad]; the word for row r and
 *          128-wide K slice g holds in byte j the factor of the 1x32 block
 *          4g + j, and sits at index g * R_pad + (r & ~127) + 4 * (r % 32) +
 *          (r % 128) / 32.  Words of padding rows are written as 127 bytes.
 *          Size: 4 * (K/128) * R_pad bytes.
 */
FP8_API int fp8_quantize_mx(const void *x, int in_dt, int64_t R, int64_t K, int fmt,
                    const float *amax, float *global_out, uint8_t *q, uint32_t *local,
                    fp8_stream_t stream);

/* ---------------------------------- quantize mx, per-row global factor --
 * The two-level scheme with the global factor of step 2 taken per row (the
 * page's garbled extent "整个 _ 范围" read per row; [MOSS] 4): row r's
 * S_r = fl32(max |x[r,:]| / MAX) (= max over its 1x32 blocks of s_i) and its
 * local factors r_i = 2^ceil(log2(s_i / S_r)).  fp8_amax_rows gives the row
 * amaxes; fp8_quantize_mx_rows quantizes with them and writes S_r to
 * global_out[r]; the codes and local words have fp8_quantize_mx's layout.
 *   amax_out / amax_rows / global_out  device fp32 [R].  K % 8 == 0 for
 *   fp8_amax_rows, K % 128 == 0 for fp8_quantize_mx_rows.
 */
FP8_API int fp8_amax_rows(const void *x, int in_dt, int64_t R, int64_t K, float *amax_out,
                          fp8_stream_t stream);
FP8_API int fp8_quantize_mx_rows(const void *x, int in_dt, int64_t R, int64_t K, int fmt,
                                 const float *amax_rows, float *global_out, uint8_t *q,
                                 uint32_t *local, fp8_stream_t stream);

/* ------------------------------------------------- quantize mx, one level --
 * fp8_quantize_mx1: plain MXFP8 ([MOSS] 1): every 32 consecutive values of a
 * row share one power-of-two scale, the smallest not below amax_i / MAX
 * (byte e + 127, e clamped to [-127, 127]; byte 127 for an all-zero block),
 * and the block is quantized with it.  The output layout is fp8_quantize_mx's
 * (codes + packed E8M0 words), so fp8_gemm_mx contracts it with global
 * factors of 1.0; global_out (nullable, device fp32) receives 1.0 for that.
 */
FP8_API int fp8_quantize_mx1(const void *x, int in_dt, int64_t R, int64_t K, int fmt,
                     float *global_out, uint8_t *q, uint32_t *local, fp8_stream_t stream);

/* ------------------------------------------- quantize 32x32 blocks --
 * fp8_quantize_block32: weight blocks of 32 x 32 with UE8M0 scales ([HF] 八:
 * weight_block_size is configurable; 七: the scale amax / MAX is rounded UP
 * to a power of two and the block is quantized with the rounded scale).
 * Block (i, j) covers rows [32i, 32i + 32) and columns [32j, 32j + 32) of
 * w [N, K]; its exponent e = ceil(log2(fl32(amax / MAX))) clamped to
 * [-127, 127] (byte 127 for an all-zero block).
 *   w       [N, K] bf16 or fp32, 16-byte aligned; K % 128 == 0.
 *   q       [N, K] uint8 codes, 16-byte aligned.
 *   scales  nullable; uint8 [ceil(N/32), K/32] block bytes.
 *   local   every row's block byte for each 1x32 piece, in fp8_quantize_mx's
 *           packed E8M0 word layout (R = N; padding rows hold 127 bytes), so
 *           that fp8_gemm_mx contracts these weights with fp8_quantize_mx1
 *           activations (both global factors 1.0).  16-byte aligned,
 *           4 * (K/128) * R_pad bytes.
 */
FP8_API int fp8_quantize_block32(const void *w, int in_dt, int64_t N, int64_t K, int fmt,
                                 uint8_t *q, uint8_t *scales, uint32_t *local,
                                 fp8_stream_t stream);

/* ------------------------------ (32, 32) weight blocks, FP32 scales --
 * The configurable weight_block_size of [HF] 八 at (32, 32) with the default
 * float scales ([HF] 四 scale_fmt): the activations go in 1 x 32 groups.
 *
 * fp8_quantize_token_group32: fp8_quantize_token_group with 1 x 32 groups:
 *   scales GROUP-MAJOR [ceil(K/32), M] (fp32 amax/MAX, 1.0 for an all-zero
 *   group; or UE8M0 bytes as there).  x [M, K], K % 16 == 0.
 * fp8_quantize_block32_f32: 32 x 32 weight blocks with fp32 scales:
 *   scales [ceil(N/32), K/32] = fl32(block amax / MAX) (1.0 for an all-zero
 *   block); each block divided by its own scale.  w [N, K], K % 32 == 0.
 * fp8_gemm_group32: C[m,n] = sum_g sa[g,m] * sb[n/32, g] * sum_{k in g} a.b
 *   over 32-wide K groups g; E4M3 codes a [M, K], b [N, K] with the scales
 *   above; bf16 output c [M, ldc].  K % 128 == 0.  Every K=32 MMA is
 *   contracted into its own tensor-memory buffer and promoted on the CUDA
 *   cores with its two scales (a promotion per 32-deep K step, four times as
 *   many as the 128-wide groups of fp8_gemm_group).
 */
FP8_API int fp8_quantize_token_group32(const void *x, int in_dt, int64_t M, int64_t K, int fmt,
                                       int sfmt, uint8_t *q, void *scales, fp8_stream_t stream);
FP8_API int fp8_quantize_block32_f32(const void *w, int in_dt, int64_t N, int64_t K, int fmt,
                                     uint8_t *q, float *scales, fp8_stream_t stream);
FP8_API int fp8_gemm_group32(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb,
                             int64_t M, int64_t N, int64_t K, void *c, int64_t ldc,
                             fp8_stream_t stream);

/* --------------------------------------------------- dequantize block --
 * fp8_dequantize_block: out[n,k] = decode(q[n,k]) * scale of block
 * (n/128, k/128), rounded to bf16 ([HF] 五: dequantize=True folds the block
 * scales back into bf16 weights).  q [N, K] codes (8-byte aligned), scales as
 * written by fp8_quantize_block (fp32 or UE8M0 bytes), out [N, K] bf16
 * (16-byte aligned).  K % 16 == 0.  The product is formed in fp32.
 */
FP8_API int fp8_dequantize_block(const uint8_t *q, int fmt, const void *scales, int sfmt,
                                 int64_t N, int64_t K, void *out, fp8_stream_t stream);

/* ------------------------------------------------------ GEMM, per tensor --
 * fp8_gemm_tensor: C = (sa * sb) * (A_q . B_q^T) with FP32 accumulation in
 * TMEM and the scales applied in the epilogue ([Flax] 2.2: dot with
 * preferred_element_type = f32, then dequantize by a_scale * b_scale; [Nano]
 * "实现": out_dtype bf16).
 *   a  [M, K] uint8 codes of format fa; b [N, K] codes of format fb.
 *      E4M3 x E4M3 (forward) and E5M2 x E4M3 (gradient GEMMs) are the uses;
 *      every E4M3/E5M2 pairing is accepted.
 *   sa, sb  device fp32 scalars (dequant scales).
 *   K % 16 == 0; a, b 16-byte aligned.  M, N >= 1 (ragged tiles are masked).
 *   out_dt  FP8_OUT_F32 or FP8_OUT_BF16 (RNE); c [M, ldc] row-major,
 *           aligned to its element size, ldc >= N.  (A 16-byte aligned c with
 *           ldc * elemsize % 16 == 0 takes the vector-store path.)
 *   accumulate  0: C = result.  1 (FP8_OUT_F32 only): C += result.
 */
FP8_API int fp8_gemm_tensor(const uint8_t *a, int fa, const uint8_t *b, int fb, const float *sa,
                    const float *sb, int64_t M, int64_t N, int64_t K, int out_dt, void *c,
                    int64_t ldc, int accumulate, fp8_stream_t stream);

/* ------------------------------------------- GEMM, per tensor, grouped --
 * fp8_gemm_tensor_grouped: `count` independent per-tensor GEMMs in one call,
 * each computed as fp8_gemm_tensor would (same bound), with a storage layout
 * per operand.  Up to 4 problems whose shapes suit the CTA-pair path run as
 * ONE persistent launch over all their tiles (longest K first), which pays
 * the kernel prologue, pipeline fill and tail once instead of per GEMM --
 * e.g. the forward and both backward GEMMs of a linear layer once their
 * operands are quantized ([Nano] "实现": three GEMMs).  Otherwise the
 * problems run one after another on `stream`.
 *   problems  HOST array of `count` descriptors (read during the call only);
 *             the pointers inside are device pointers as for fp8_gemm_tensor.
 *   a_layout, b_layout  FP8_K_MAJOR (a [M, K], b [N, K], as fp8_gemm_tensor)
 *             or FP8_MN_MAJOR (a [K, M], b [K, N]: the row-major codes of a
 *             row-major tensor used transposed, so that dx = g W and
 *             dW = g^T x read the codes of g, W and x without a transposed
 *             copy).  An MN-major operand needs its row count (M or N) to be
 *             a multiple of 16; K % 16 == 0 is needed only while an operand
 *             is K-major.  FP8_ERR_MISALIGNED otherwise.
 *   No output may overlap another problem's output or inputs.
 *   A group with an epilogue variant (adamw or swiglu) runs as one CTA-pair
 *   launch whatever the shapes (ragged tiles are masked; no split K, even for
 *   small M) and holds at most 4 problems (FP8_ERR_UNSUPPORTED otherwise).
 */
/* Epilogue variants of a grouped per-tensor problem (fp8_gemm_tensor_grouped;
 * CTA-pair path only).  Both fold element-wise work of the FP8 training step
 * into the GEMM's epilogue, which reads the accumulator from tensor memory
 * instead of a stored result from HBM.  Not described on the pages (the
 * SwiGLU MLP and AdamW around the FP8 GEMMs are support arithmetic); the
 * values are exactly those of the standalone calls named below. */

/* AdamW epilogue: the problem's fp32 result G = sa*sb*A*B^T is the gradient of
 * the parameters p [M, N] (row pitch ldc) and is NOT stored (c may be null);
 * instead each element is updated as fp8_adamw_multi would update it with
 * gradient G at step t = step[0] (device int64, read only; advance it first,
 * e.g. fp8_adamw_multi with count 0).  p, m, v fp32 16-byte aligned, p_bf16
 * (nullable) bf16 8-byte aligned, ldc % 4 == 0.  The problem must have
 * out_dt FP8_OUT_F32, accumulate 0 and no bias. */
typedef struct {
  float *p, *m, *v;
  void *p_bf16;
  const int64_t *step;
  double lr, beta1, beta2, eps, weight_decay;
} fp8_adamw_epilogue_t;

/* Gated SwiGLU epilogue (h = A B^T, u = A B_up^T, a = silu(h) * u): the pair
 * computes h and u for the same output columns (B = W1 codes, b_up = W3 codes
 * in the same layout and format, scale sb_up) and writes c <- bf16(h) (the
 * problem's output, FP8_OUT_BF16), u <- bf16(u), q <- codes of
 * a = bf16(silu(h) u) divided by scale[0] (format fmt), amax[0] <- max |a|
 * (cleared by the call) -- what fp8_swiglu_forward_quantize gives for the
 * stored h and u.  c, u, q [M, N] with row pitch ldc (elements; q in bytes),
 * 16-byte aligned, ldc % 16 == 0, N % 32 == 0; no bias, no accumulate. */
typedef struct {
  const uint8_t *b_up;
  const float *sb_up;
  void *u;
  uint8_t *q;
  int fmt;
  const float *scale;
  float *amax;
} fp8_swiglu_epilogue_t;

typedef struct {
  const uint8_t *a; /* codes of format fa: [M, K] (K-major) or [K, M] (MN-major) */
  const uint8_t *b; /* codes of format fb: [N, K] (K-major) or [K, N] (MN-major) */
  const float *sa;  /* device fp32 dequant scale of a */
  const float *sb;  /* device fp32 dequant scale of b */
  int64_t M, N, K;
  int fa, fb;
  int out_dt;     /* FP8_OUT_F32 or FP8_OUT_BF16 */
  int accumulate; /* 1: C += result (FP8_OUT_F32 only) */
  void *c;        /* [M, ldc] row-major */
  int64_t ldc;
  int a_layout;   /* fp8_layout_t */
  int b_layout;   /* fp8_layout_t */
  const float *bias; /* nullable device fp32 [N]: C = result + bias[n] ([Nano]
                        "实现": the linear's bias; added in fp32 before the
                        output cast; with accumulate, C += result + bias) */
  const fp8_adamw_epilogue_t *adamw;   /* nullable HOST pointer (read during the call) */
  const fp8_swiglu_epilogue_t *swiglu; /* nullable HOST pointer (read during the call) */
} fp8_gemm_problem_t;

FP8_API int fp8_gemm_tensor_grouped(const fp8_gemm_problem_t *problems, int count,
                                    fp8_stream_t stream);

/* ---------------------------------------------------- GEMM, per K group --
 * fp8_gemm_group: C[m,n] = sum_g sa[g,m] * sb[n/128, g] * sum_{k in g} a.b
 * ([HF] 一: 1x128 activation groups times 128x128 weight blocks), output
 * bf16.  The per-group scales are applied in the main loop.
 *   a  [M, K] E4M3 codes, sa GROUP-MAJOR [K/128, M] (fp8_quantize_token_group).
 *   b  [N, K] E4M3 codes, sb [ceil(N/128), K/128] (fp8_quantize_block).
 *   sfmt FP8_SCALE_F32: fp32 scales, partial sums promoted per 128-K group on
 *        the CUDA cores.  FP8_SCALE_UE8M0: byte scales, applied by the tensor
 *        core as block scale factors (no promotion); with 1-128 rows they
 *        are promoted like fp32 scales (exact powers of two).
 *   K % 128 == 0.  c [M, ldc] bf16 as for fp8_gemm_tensor.
 *   With 1-128 rows the call runs the few-row kernel (FP8_OPT_GEMM_SKINNY),
 *   launched with programmatic stream serialization: it may start before the
 *   previous kernel on `stream` ends, and then reads and writes nothing that
 *   kernel may write until it has completed.  Every per-group GEMM launch and
 *   fp8_quantize_token_group (/32) are launched that way.
 */
FP8_API int fp8_gemm_group(const uint8_t *a, const void *sa, const uint8_t *b, const void *sb,
                   int sfmt, int64_t M, int64_t N, int64_t K, void *c, int64_t ldc,
                   fp8_stream_t stream);

/* ------------------------------------- GEMM, per K group, no allocation --
 * fp8_gemm_group_noalloc: the per-K-group GEMM of fp8_gemm_group (same
 * arguments, same definition, same bound) for callers that cannot allocate
 * device memory.  The pages have no counterpart to this entry point; it
 * exists for this library's users.  Its result agrees with fp8_gemm_group's
 * within the GEMM bound, not bit for bit: it always runs the general
 * tensor-core per-group kernel, while fp8_gemm_group runs 1-128 rows on its
 * few-row kernel and converts UE8M0 scales to block-scale words for
 * M > 128.
 *
 * Why: fp8_gemm_group allocates device memory on first use for some shapes
 * (the E8M0-word buffer of UE8M0 scales at M > 128).  Some callers cannot
 * let a library do that: runtimes that reserve all device memory up front in
 * their own pool (an inference server with a fixed memory budget), and code
 * that must never stall on the allocator (cudaMalloc and cudaFree may
 * synchronize the device).  This entry point calls no cudaMalloc, cudaFree
 * or other allocating routine: where it splits K over CTAs for small M, its
 * fp32 partial sums and per-tile counters live in one array compiled into
 * the library (64 KiB of counters + 8 MiB of fp32 partials, 256-byte
 * aligned), which every GPU that loads the library holds until the process
 * exits.  The caller still passes the inputs and the output.
 *
 * Limits and rules:
 *   - A shape whose split-K partials need more than 8 MiB (or more than 16384
 *     output tiles of counters) is rejected with FP8_ERR_SCRATCH_LIMIT; shapes
 *     that need no split run without the array.
 *   - The first call on each device looks up the array's device address (and
 *     does the library's per-device set-up); make that first call before any
 *     stream capture.
 *   - Every call on a device shares the one array, and it keeps the last
 *     call's contents; each call clears the counters it uses on its stream
 *     before the kernel runs.  Calls that overlap on the GPU (different
 *     streams, or concurrent graph branches) race on the array and give wrong
 *     results: serialize them.
 */
FP8_API int fp8_gemm_group_noalloc(const uint8_t *a, const void *sa, const uint8_t *b,
                                   const void *sb, int sfmt, int64_t M, int64_t N, int64_t K,
                                   void *c, int64_t ldc, fp8_stream_t stream);

/* fp8_gemm_group_bias: fp8_gemm_group plus an epilogue bias, C[m,n] =
 * result + bias[n] (bias: device fp32 [N], added in fp32 before the bf16
 * cast, in every path: promotion, block-scaled, split K).  bias == NULL is
 * fp8_gemm_group. */
FP8_API int fp8_gemm_group_bias(const uint8_t *a, const void *sa, const uint8_t *b, const void *sb,
                                int sfmt, int64_t M, int64_t N, int64_t K, const float *bias,
                                void *c, int64_t ldc, fp8_stream_t stream);

/* fp8_gemm_mx_rows: fp8_gemm_mx with per-row global factors (operands from
 * fp8_quantize_mx_rows): C[m,n] = (ga[m] * gb[n]) * sum_i r_a r_b sum a.b;
 * ga device fp32 [M], gb device fp32 [N]. */
FP8_API int fp8_gemm_mx_rows(const uint8_t *a, const uint32_t *la, const float *ga,
                             const uint8_t *b, const uint32_t *lb, const float *gb, int64_t M,
                             int64_t N, int64_t K, int out_dt, void *c, int64_t ldc,
                             fp8_stream_t stream);

/* ------------------------------------- GEMM, per K group, MoE experts --
 * fp8_gemm_group_experts: the per-K-group GEMM of a mixture-of-experts layer
 * whose token rows are grouped by expert ([HF] 一 and 六 6.4: FP8Experts,
 * 128x128 weight blocks per expert; 七: UE8M0 scales).  Rows
 * [offsets[e], offsets[e+1]) of A are the tokens routed to expert e, and for
 * such a row m
 *   C[m,n] = sum_g sa[g,m] * sb[e][n/128, g] * sum_{k in g} a[m,k] b[e][n,k].
 *   a        [M, K] E4M3 codes, sa [K/128, M] (fp8_quantize_token_group)
 *   b        [E, N, K] E4M3 codes, expert-major: expert e's [N, K] block
 *            quantized as by fp8_quantize_block
 *   sb       [E, ceil(N/128), K/128] scales (fp32 or UE8M0 bytes per sfmt)
 *   offsets  DEVICE int32 [E + 1]: 0 = offsets[0] <= ... <= offsets[E] = M;
 *            segments of any size, empty experts allowed.  Read by the
 *            kernel: the host does not check them (a tile never spans two
 *            experts; rows outside [0, M) are never loaded or stored).
 *   experts  E, 1 <= E <= 256.  c [M, ldc] bf16.  K % 128 == 0.
 * One persistent launch over all experts' tiles (each expert's row range
 * split into 128-row tiles); no split K.
 */
FP8_API int fp8_gemm_group_experts(const uint8_t *a, const void *sa, const uint8_t *b,
                                   const void *sb, int sfmt, const int32_t *offsets, int experts,
                                   int64_t M, int64_t N, int64_t K, void *c, int64_t ldc,
                                   fp8_stream_t stream);

/* ----------------------------------------------------- GEMM, two level --
 * fp8_gemm_mx: C = S_a * S_b * sum_i r_a[m,i] r_b[n,i] sum_{k in i} a.b
 * ([MOSS] 4, step 4): the E8M0 local factors are block scale factors of the
 * MMA (kind::mxf8f6f4, one per 1x32), the FP32 global factors are applied
 * once in the epilogue.
 *   a [M, K], b [N, K] E4M3 codes; la, lb local factors in the layout written
 *   by fp8_quantize_mx (R_pad = M or N rounded up to 128); ga, gb device fp32
 *   global factors.  K % 128 == 0.  out_dt / c / ldc as for fp8_gemm_tensor.
 */
FP8_API int fp8_gemm_mx(const uint8_t *a, const uint32_t *la, const float *ga, const uint8_t *b,
                const uint32_t *lb, const float *gb, int64_t M, int64_t N, int64_t K,
                int out_dt, void *c, int64_t ldc, fp8_stream_t stream);

/* -------------------------------------------------- delayed-state update --
 * fp8_delayed_state_update: one amax-history step of delayed scaling
 * ([Flax] 2.3 compute_amax_history / update_fp8_meta), on device, no host
 * synchronisation.  In order:
 *   1. hist <- roll(hist, -1); hist[0] <- amax_cur[0]   (element 0 is newest)
 *   2. m = max(hist); scale[0] <- fl32(m / MAX) if m > 0 and finite, else
 *      scale[0] is kept.
 * hist [L] fp32 (L >= 1), scale [1] fp32, amax_cur [1] fp32 (the fused amax
 * fp8_quantize_tensor wrote for this step).  After the call scale[0] is the
 * scale the NEXT step quantizes with; starting from the guide's initial state
 * (zeros, 1.0) this reproduces in_q's order exactly (the guide computes the
 * scale from the history before pushing the current amax, [Flax] 2.3).
 */
FP8_API int fp8_delayed_state_update(float *hist, float *scale, const float *amax_cur, int64_t L,
                             int fmt, fp8_stream_t stream);

/* fp8_delayed_state_update_multi: the step above for `count` (1..16)
 * independent histories in one launch (a training step keeps one per GEMM
 * operand).  Each item's hist, scale, amax_cur, L and fmt mean what the
 * arguments of fp8_delayed_state_update mean, with the same checks.  The
 * items' hist ranges and scale words must not overlap each other
 * (INVALID_ARG); an item's amax_cur may be another item's (it is only
 * read).  The same results as `count` calls of fp8_delayed_state_update. */
typedef struct {
  float *hist;            /* [L] fp32, element 0 newest */
  float *scale;           /* [1] fp32 */
  const float *amax_cur;  /* [1] fp32 */
  int64_t L;              /* 1 .. 32768 */
  int fmt;                /* FP8_E4M3 / FP8_E5M2 */
} fp8_delayed_item_t;
FP8_API int fp8_delayed_state_update_multi(const fp8_delayed_item_t *items, int count,
                                           fp8_stream_t stream);

/* ------------------------------------------- automatic weight scaling --
 * fp8_auto_weight_scale: MOSS automatic scaling ([MOSS] 5, eq. 10): the scale
 * of a weight t optimizer steps after its last max-reduction is predicted,
 * without reading the weight, as
 *     scale_out[0] = fl32(fl32(amax0[0] + fl32(lr * t)) / MAX)
 * (an Adam step moves each weight by about lr at most).  amax0: device fp32,
 * the weight's amax at the last max-reduction (fp8_amax, every ~500 steps);
 * lr * t is formed in double on the host.  t >= 0.
 */
FP8_API int fp8_auto_weight_scale(const float *amax0, int64_t t, double lr, int fmt,
                                  float *scale_out, fp8_stream_t stream);

/* -------------------------------------------- SwiGLU / AdamW (support) --
 * Support kernels of the FP8 SwiGLU training step.  Not described on the
 * pages; plain definitions: silu(z) = z / (1 + exp(-z)) in fp32.
 * fp8_swiglu_forward: a = silu(h) * u (bf16 in, bf16 out), n elements.
 * fp8_swiglu_backward: dh = da * u * silu'(h), du = da * silu(h), bf16.
 * fp8_adamw_step: decoupled-weight-decay Adam on fp32 master weights p with
 *   moments m, v (fp32), gradient g (fp32); writes the bf16 copy p_bf16
 *   (nullable).  step counts from 1.  All buffers 16-byte aligned.  The
 *   hyperparameters are doubles: 1 - beta and the bias corrections are formed
 *   in double before the kernel sees them in fp32.
 */
FP8_API int fp8_swiglu_forward(const void *h, const void *u, void *a, int64_t n, fp8_stream_t stream);
FP8_API int fp8_swiglu_backward(const void *da, const void *h, const void *u, void *dh, void *du,
                        int64_t n, fp8_stream_t stream);
FP8_API int fp8_adamw_step(float *p, const float *g, float *m, float *v, void *p_bf16, int64_t n,
                   int64_t step, double lr, double beta1, double beta2, double eps,
                   double weight_decay, fp8_stream_t stream);

/* ------------------------------- SwiGLU fused with delayed scaling --
 * With delayed scaling the quantization scale of a tensor is known before
 * the tensor is formed ([Flax] 2.3: in_q quantizes with the scale the
 * previous step's amax history left and records the current amax), so the
 * SwiGLU passes can quantize their outputs as they produce them.  The values
 * are exactly those of fp8_swiglu_forward / _backward (the same bf16
 * rounding), and the codes and amax exactly those fp8_quantize_tensor would
 * give for that bf16 tensor with `scale` and `amax_out`: the bf16 tensor is
 * simply never written to memory.
 *
 * fp8_swiglu_forward_quantize: a = bf16(silu(h) * u); q = codes of a / scale
 *   (fmt), amax_out = max |a| (nullable; cleared first; must not alias scale).
 * fp8_swiglu_backward_quantize: dh, du as fp8_swiglu_backward; q_dh, q_du =
 *   their codes under scale_dh, scale_du (both in format fmt, E5M2 for
 *   gradients, [Flax] 3.3); amax_dh, amax_du = max |dh|, max |du| (both null
 *   or both set, distinct from each other and from the scales).
 * n elements, n % 8 == 0; h, u, da bf16, 16-byte aligned; q's 16-byte aligned.
 * n == 0 writes only the amaxes (0); the other pointers may then be null.
 */
FP8_API int fp8_swiglu_forward_quantize(const void *h, const void *u, int64_t n, int fmt,
                                        const float *scale, uint8_t *q, float *amax_out,
                                        fp8_stream_t stream);
FP8_API int fp8_swiglu_backward_quantize(const void *da, const void *h, const void *u, int64_t n,
                                         int fmt, const float *scale_dh, const float *scale_du,
                                         uint8_t *q_dh, uint8_t *q_du, float *amax_dh,
                                         float *amax_du, fp8_stream_t stream);

/* fp8_adamw_multi: one AdamW step (as fp8_adamw_step) over `count` (0..8)
 * parameter tensors in one launch, with the step number kept on the device
 * (*step: device int64, 8-byte aligned; bias corrections 1 - beta^t formed in
 * double on the device).  advance = 1: the call first increments *step and
 * the update uses the incremented value as t; advance = 0: the update uses
 * t = *step as it stands (for the other updates of the same step, e.g. on a
 * second stream).  A captured training step therefore advances t on every
 * replay.  Start *step at 0 for a fresh optimizer.  count == 0 with
 * advance = 1 only advances the counter (items may be null): for updates
 * done later in the step, by further calls with advance = 0 or by GEMM
 * epilogues (fp8_adamw_epilogue_t), which read t without advancing it.
 *   items  HOST array of `count` descriptors (read during the call only);
 *          per item p, g, m, v fp32 [n] and p_bf16 (nullable) bf16 [n], all
 *          device, 16-byte aligned (p_bf16 8-byte), n % 4 == 0; empty items
 *          (n == 0) may have null pointers.
 *          q (nullable): the item's next delayed-scaling quantization done
 *          here, on the updated weights ([Flax] 2.3: the weight is quantized
 *          with the scale its history left): q [n] receives the codes of
 *          bf16(p) divided by q_scale[0] (format q_fmt), exactly what
 *          fp8_quantize_tensor(bf16(p), scale = q_scale) gives, and
 *          q_amax[0] (nullable) max |bf16(p)| (cleared by the call), the
 *          amax that the weight's history then takes.  q 4-byte aligned;
 *          q_scale required with q; q_amax must not alias q_scale or another
 *          item's q_amax. */
typedef struct {
  float *p;
  const float *g;
  float *m;
  float *v;
  void *p_bf16;
  int64_t n;
  uint8_t *q;
  const float *q_scale;
  float *q_amax;
  int q_fmt;
} fp8_adamw_item_t;
FP8_API int fp8_adamw_multi(const fp8_adamw_item_t *items, int count, int64_t *step,
                            int advance, double lr, double beta1, double beta2, double eps,
                            double weight_decay, fp8_stream_t stream);

/* ---------------------------------------------------------------- status --
 * fp8_status_string: static text for a status code.
 * fp8_get_last_device_error: synchronises `stream`, then returns (and clears)
 * the first device-side error recorded since the last read: 0 for none,
 * FP8_ERR_TIMEOUT when a bounded wait expired; *where_out (nullable) receives
 * a small code naming the wait (1 producer, 2 MMA, 3 epilogue).
 * fp8_version: library version string.
 */
FP8_API const char *fp8_status_string(int status);
FP8_API int fp8_get_last_device_error(int *where_out, fp8_stream_t stream);
FP8_API const char *fp8_version(void);

/* fp8_set_option: process-wide switches (not thread-safe against concurrent
 * GEMM calls).
 *   FP8_OPT_GEMM_CTA_PAIRS: 1 (default) lets fp8_gemm_tensor run large shapes
 *     on CTA pairs (tcgen05 cta_group::2, 256 x 256 tiles) and fp8_gemm_group
 *     with FP32 scales run them on pairs of 256 x 128 tiles; 0 keeps every
 *     GEMM on single-CTA tiles.  Results agree within the GEMM bound.
 *   FP8_OPT_WAIT_LIMIT_US: bound, in microseconds, of every device-side
 *     mbarrier wait of later GEMM launches (default 2,000,000).  A wait that
 *     runs out records FP8_ERR_TIMEOUT in the device error word and the
 *     kernel exits cleanly (output undefined).  Small values exist to test
 *     that path.
 *   FP8_OPT_GEMM_MULTICAST: 1 (default) runs the per-group and block-scaled
 *     GEMMs that use 128-wide tiles (K-major weights, no split K) as
 *     clusters of two CTAs on vertically adjacent tiles that share each
 *     weight box through TMA multicast; 0 gives every CTA its own copy.
 *     Same results.
 *   FP8_OPT_GEMM_TMA_STORE: 1 lets the CTA-pair per-tensor GEMM write C
 *     through shared memory with TMA stores (when c and ldc allow 16-byte
 *     vectors and accumulate is 0); 0 (default) keeps plain per-thread row
 *     stores, which measured faster.  Same bytes.
 *   FP8_OPT_GEMM_FEW_ROWS: 1 runs fp8_gemm_group / _group_bias with a
 *     single activation row on the CUDA cores as a stream over the weights;
 *     0 (default) keeps it on the tensor cores (the few-row kernel of
 *     FP8_OPT_GEMM_SKINNY, which measured faster inside CUDA graphs).
 *     Results agree within the GEMM bound.
 *   FP8_OPT_GEMM_BAND_ROWS: height, in 256-row tiles, of the bands in which
 *     the CTA-pair per-tensor GEMM walks its output tiles column by column
 *     (1..4096, default 8): taller bands read each B column block from DRAM
 *     fewer times, at the price of a larger A working set in L2.  Same
 *     results.
 *   FP8_OPT_GEMM_SKINNY: 1 (default) runs fp8_gemm_group / _group_bias with
 *     1 to 128 activation rows (one row only while FP8_OPT_GEMM_FEW_ROWS is
 *     0) on the few-row tensor-core kernel: 128 weight rows per tile on the
 *     MMA's M side, the activation rows padded to 16, 32 or 64 on its N
 *     side (65-128 rows as two 64-row halves of CTAs), K split over a
 *     thread-block cluster, launched so that it may
 *     start before the previous kernel in the stream ends; 0 keeps them on
 *     the general per-group kernel.  Results agree within the GEMM bound. */
typedef enum {
  FP8_OPT_GEMM_CTA_PAIRS = 1,
  FP8_OPT_WAIT_LIMIT_US = 2,
  FP8_OPT_GEMM_MULTICAST = 3,
  FP8_OPT_GEMM_TMA_STORE = 4,
  FP8_OPT_GEMM_FEW_ROWS = 5,
  FP8_OPT_GEMM_BAND_ROWS = 6,
  FP8_OPT_GEMM_SKINNY = 7
} fp8_option_t;
FP8_API int fp8_set_option(int option, int value);

#ifdef __cplusplus
}
#endif

#endif /* FP8GEMM_H */
