// Amax and quantization kernels (HBM-bound, CUDA cores).
//
// Every kernel reads its input with 16-byte vector loads, reduces |x| with
// warp shuffles on order-preserving uint32 keys (exact: max is order
// independent), and casts on store with cvt.rn.satfinite after the
// fl32(x / s) division and the +-MAX clip of the Flax guide's `quantize`
// (section 2.2).  The division is the correctly rounded quotient formed from
// one reciprocal per scale (div_by_scale in common.cuh).
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "quant_common.cuh"

namespace fp8k {

// ------------------------------------------------------------------ amax --
// One wave of persistent CTAs (2 x 512 threads per SM) streams the tensor
// with batches of eight independent 16-byte loads per thread.
template <typename T>
__global__ void __launch_bounds__(512, 2) amax_kernel(const T *__restrict__ x, int64_t n,
                                                      uint32_t *__restrict__ out) {
  uint32_t key_a = 0, key_b = 0;
  const int64_t nvec = n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < nvec;
       base += 8 * stride) {
    // loads are unconditional (index clamped in range) so that all eight are
    // in flight at once; a clamped load repeats the last vector, which leaves
    // the max unchanged
    Raw8<T> raw[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t i = base + u * stride;
      raw[u].load_stream(x + (i < nvec ? i : nvec - 1) * 8);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) raw[u].max_abs(key_a, key_b);
  }
  uint32_t key = Raw8<T>::merge_keys(key_a, key_b);
  for (int64_t i = nvec * 8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    key = max(key, abs_key(load1(x + i)));
  block_max_to(key, out);
}

// ------------------------------------------------------- quantize tensor --
__device__ __forceinline__ float resolve_scale(const float *amax_in, const float *scale_in,
                                               float mx) {
  return amax_in != nullptr ? scale_from_amax(*amax_in, mx) : *scale_in;
}

// Row-major output only, in windows of 1024 elements: lane l of a warp owns
// elements [32 l, 32 l + 32) of a window (four adjacent 16-byte loads for
// bf16), and a warp takes kU windows at once (w, w + W, ..., W warps in the
// grid), issuing all their loads before it converts any; the lane's 32 codes
// go out as two 16-byte stores.  (Grid-stride 16-byte vectors with the next
// batch's loads issued before the current one's conversion measured 10%
// slower than this layout.)  kFast selects the reciprocal-based quotient
// (ScaleDiv), checked once per launch.  The fused amax takes |x| from the raw
// words (two bf16 keys per instruction).
template <typename T, int F, bool kAmax, bool kFast>
__device__ __forceinline__ void quant_tensor_body(const T *__restrict__ x, int64_t n,
                                                  const ScaleDiv &d, uint8_t *__restrict__ q,
                                                  uint32_t &key) {
  constexpr int kU = sizeof(T) == 2 ? 2 : 1;
  const int64_t nvec = n / 8;  // n % 8 == 0 (the row length is)
  const int64_t nwin = (nvec + 127) / 128;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t l = lane_id();
  uint32_t key_a = 0, key_b = 0;
  for (int64_t w0 = warp; w0 < nwin; w0 += kU * nwarps) {
    Raw8<T> r[kU][4];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t v0 = (w0 + u * nwarps) * 128 + l * 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (v0 + i < nvec)
          r[u][i].load_stream(x + (v0 + i) * 8);
        else
          r[u][i].zero();
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (w0 + u * nwarps >= nwin) break;  // warp-uniform
      const int64_t v0 = (w0 + u * nwarps) * 128 + l * 4;
      uint2 c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if constexpr (sizeof(T) == 2 && kFast) {
          // bf16 on the fast path: quotients of |x| clamped, signs from the
          // words; the same two-halfword key as max_abs (unused without kAmax)
          c[i] = quant_bf16x8<F>(r[u][i].w[0], d, key_a);
        } else {
          if (kAmax) r[u][i].max_abs(key_a, key_b);  // zero-filled vectors add nothing
          float v[8], y[8];
          r[u][i].decode(v);
          d.div8<kFast>(v, y);
          c[i] = pack8<F>(y);
        }
      }
      uint2 *dst = reinterpret_cast<uint2 *>(q) + v0;
      if (v0 + 4 <= nvec) {
        reinterpret_cast<uint4 *>(dst)[0] = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
        reinterpret_cast<uint4 *>(dst)[1] = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (v0 + i < nvec) dst[i] = c[i];
      }
    }
  }
  if (kAmax) key = max(key, Raw8<T>::merge_keys(key_a, key_b));
}

template <typename T, int F, bool kAmax>
__global__ void __launch_bounds__(256, 3)
    quant_tensor_kernel(const T *__restrict__ x, int64_t n, const float *amax_in,
                        const float *scale_in, float *scale_out, uint8_t *__restrict__ q,
                        uint32_t *amax_out) {
  const float mx = fmt_max(F);
  const float s = resolve_scale(amax_in, scale_in, mx);
  if (scale_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *scale_out = s;
  const ScaleDiv d(s);
  uint32_t key = 0;
  if (d.fast)
    quant_tensor_body<T, F, kAmax, true>(x, n, d, q, key);
  else
    quant_tensor_body<T, F, kAmax, false>(x, n, d, q, key);
  if (kAmax) block_max_to(key, amax_out);
}

// Row-major output plus the transposed copy q_t [cols, rows], in 128 x 128
// tiles staged through shared memory.  The 8-byte chunk c of tile row r is
// stored at chunk c ^ (r / 8), so that both the row-wise writes and the 8x8
// byte-block reads of the transpose are free of bank conflicts.
constexpr int kTT = 128;
constexpr int kTPitch = kTT;
__device__ __forceinline__ int tchunk(int r, int c8) { return ((c8 ^ (r >> 3)) & 15) * 8; }

// 4x4 byte transpose: byte j of word i -> byte i of word j.
__device__ __forceinline__ void transpose4x4(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                             uint32_t (&o)[4]) {
  const uint32_t ab01 = __byte_perm(a, b, 0x5140), cd01 = __byte_perm(c, d, 0x5140);
  const uint32_t ab23 = __byte_perm(a, b, 0x7362), cd23 = __byte_perm(c, d, 0x7362);
  o[0] = __byte_perm(ab01, cd01, 0x5410);
  o[1] = __byte_perm(ab01, cd01, 0x7632);
  o[2] = __byte_perm(ab23, cd23, 0x5410);
  o[3] = __byte_perm(ab23, cd23, 0x7632);
}

// 8x8 byte transpose from four 4x4 ones: byte j of r[i] -> byte i of c[j].
__device__ __forceinline__ void transpose8x8(const uint64_t (&r)[8], uint64_t (&c)[8]) {
  uint32_t lo_top[4], lo_bot[4], hi_top[4], hi_bot[4];
  transpose4x4((uint32_t)r[0], (uint32_t)r[1], (uint32_t)r[2], (uint32_t)r[3], lo_top);
  transpose4x4((uint32_t)r[4], (uint32_t)r[5], (uint32_t)r[6], (uint32_t)r[7], lo_bot);
  transpose4x4((uint32_t)(r[0] >> 32), (uint32_t)(r[1] >> 32), (uint32_t)(r[2] >> 32),
               (uint32_t)(r[3] >> 32), hi_top);
  transpose4x4((uint32_t)(r[4] >> 32), (uint32_t)(r[5] >> 32), (uint32_t)(r[6] >> 32),
               (uint32_t)(r[7] >> 32), hi_bot);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    c[j] = (uint64_t)lo_top[j] | ((uint64_t)lo_bot[j] << 32);
    c[4 + j] = (uint64_t)hi_top[j] | ((uint64_t)hi_bot[j] << 32);
  }
}

template <typename T, int F, bool kAmax, bool kFast>
__device__ __forceinline__ void quant_tensor_t_body(const T *__restrict__ x, int64_t rows,
                                                    int64_t cols, const ScaleDiv &d,
                                                    uint8_t *__restrict__ q,
                                                    uint8_t *__restrict__ qt, uint8_t *tile,
                                                    uint32_t &key) {
  // tile counts fit 32 bits (rows, cols < 2^31 and 128-wide tiles), so the
  // tile -> (row, column) split is a 32-bit division, once per tile
  const uint32_t tiles_c = (uint32_t)((cols + kTT - 1) / kTT);
  const uint32_t ntiles = (uint32_t)((rows + kTT - 1) / kTT) * tiles_c;
  const int t = threadIdx.x;
  const int lc = (t & 15) * 8;
  auto tile_origin = [&](uint32_t tl, int64_t &r0, int64_t &c0) {
    const uint32_t tr = tl / tiles_c;
    r0 = (int64_t)tr * kTT;
    c0 = (int64_t)(tl - tr * tiles_c) * kTT;
  };
  // Persistent CTAs loop over 128 x 128 tiles; the eight 16-byte loads of the
  // NEXT tile are issued before the current tile is processed.
  auto load_tile = [&](int64_t r0, int64_t c0, Raw8<T> (&raw)[kTT / 16]) {
    const int64_t c = c0 + lc;
#pragma unroll
    for (int pass = 0; pass < kTT / 16; ++pass) {
      const int64_t r = r0 + pass * 16 + (t >> 4);
      if (r < rows && c < cols)
        raw[pass].load_stream(x + r * cols + c);
      else
        raw[pass].zero();
    }
  };
  constexpr bool kPrefetch = sizeof(T) == 2;  // fp32 inputs: registers too tight
  Raw8<T> cur[kTT / 16], nxt[kTT / 16];
  int64_t r0 = 0, c0 = 0, nr0 = 0, nc0 = 0;
  if (blockIdx.x < ntiles) {
    tile_origin(blockIdx.x, r0, c0);
    if (kPrefetch) load_tile(r0, c0, cur);
  }
  for (uint32_t tl = blockIdx.x; tl < ntiles; tl += gridDim.x) {
    const bool has_next = tl + gridDim.x < ntiles;
    if (has_next) tile_origin(tl + gridDim.x, nr0, nc0);
    if constexpr (kPrefetch) {
      if (has_next) load_tile(nr0, nc0, nxt);
    } else {
      load_tile(r0, c0, cur);
    }
    const int64_t c = c0 + lc;
    // phase 1: quantize, row-major store, stage the codes in shared memory
#pragma unroll
    for (int pass = 0; pass < kTT / 16; ++pass) {
      const int lr = pass * 16 + (t >> 4);
      const int64_t r = r0 + lr;
      float v[8], y[8];
      cur[pass].decode(v);
      if (kAmax) {
#pragma unroll
        for (int j = 0; j < 8; ++j) key = max(key, abs_key(v[j]));
      }
      d.div8<kFast>(v, y);
      const uint2 packed = pack8<F>(y);
      if (r < rows && c < cols) *reinterpret_cast<uint2 *>(q + r * cols + c) = packed;
      *reinterpret_cast<uint2 *>(&tile[lr * kTPitch + tchunk(lr, lc >> 3)]) = packed;
    }
    __syncthreads();
    // phase 2: thread -> one 8x8 byte block; 16 threads per q_t row segment
    const int rb = t & 15, cb = t >> 4;
    uint64_t rr[8], cc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      rr[i] = *reinterpret_cast<const uint64_t *>(&tile[(rb * 8 + i) * kTPitch + tchunk(rb * 8 + i, cb)]);
    transpose8x8(rr, cc);
    const int64_t orow0 = c0 + cb * 8;  // q_t row = input column
    const int64_t ocol = r0 + rb * 8;   // q_t column = input row
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t orow = orow0 + j;
      if (orow >= cols) break;
      uint8_t *dst = qt + orow * rows + ocol;
      if (ocol + 8 <= rows && (rows & 7) == 0) {
        *reinterpret_cast<uint64_t *>(dst) = cc[j];
      } else {
        for (int i = 0; i < 8 && ocol + i < rows; ++i) dst[i] = (uint8_t)(cc[j] >> (8 * i));
      }
    }
    __syncthreads();  // the tile buffer is rewritten by the next iteration
    if constexpr (kPrefetch) {
#pragma unroll
      for (int pass = 0; pass < kTT / 16; ++pass) cur[pass] = nxt[pass];
    }
    r0 = nr0;
    c0 = nc0;
  }
}

template <typename T, int F, bool kAmax>
__global__ void __launch_bounds__(256, 2)
    quant_tensor_t_kernel(const T *__restrict__ x, int64_t rows, int64_t cols,
                          const float *amax_in, const float *scale_in, float *scale_out,
                          uint8_t *__restrict__ q, uint8_t *__restrict__ qt,
                          uint32_t *amax_out) {
  __shared__ __align__(16) uint8_t tile[kTT * kTPitch];
  const float mx = fmt_max(F);
  const float s = resolve_scale(amax_in, scale_in, mx);
  if (scale_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *scale_out = s;
  const ScaleDiv d(s);
  uint32_t key = 0;
  if (d.fast)
    quant_tensor_t_body<T, F, kAmax, true>(x, rows, cols, d, q, qt, tile, key);
  else
    quant_tensor_t_body<T, F, kAmax, false>(x, rows, cols, d, q, qt, tile, key);
  if (kAmax) block_max_to(key, amax_out);
}

// --------------------------------------------------- token group (1x128) --
// One warp per (row, 1024-wide window of K): lane l owns the 32 elements
// [32l, 32l + 32) of the window, so four lanes form a 1x128 group (lanes
// 4c..4c+3: group 8w + c of window w) and each lane forms its group's scale
// once for 32 elements.  Each warp takes kU windows at once (w, w + W, ...,
// W warps in the grid) and issues all their loads first.  (Issuing the next
// windows' loads before converting the current ones, at two CTAs per SM for
// the registers, measured slower: 24.6 against 22.5 us at M 4096, K 7168.)
//
// Launched with programmatic stream serialization: it lets the next kernel
// start at once (a GEMM that reads these codes then brings its weights into
// L2 meanwhile, and waits for this kernel before it reads anything this
// kernel writes) and waits itself for the kernel before it.
template <typename T, int F, int GS>
__global__ void __launch_bounds__(256, 3)
    quant_group_kernel(const T *__restrict__ x, int64_t M, int64_t K, int sfmt,
                       uint8_t *__restrict__ q, void *scales) {
  constexpr int kU = sizeof(T) == 2 ? 2 : 1;
  constexpr int kShift = GS == 128 ? 7 : 5;  // log2 of the group size
  launch_dependents();
  grid_dependency_wait();
  const float mx = fmt_max(F);
  const int64_t G = (K + GS - 1) / GS, wins = (K + 1023) / 1024, ntasks = M * wins;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const bool narrow = ntasks + kU * nwarps <= (int64_t)0xFFFFFFFFu;
  const uint32_t l = lane_id();
  for (int64_t base = warp; base < ntasks; base += kU * nwarps) {
    Run32<T> run[kU];
    int64_t row[kU], col[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t task = base + u * nwarps;
      int64_t w;
      split_task(task, wins, narrow, row[u], w);
      col[u] = w * 1024 + l * 32;
      if (task < ntasks)
        run[u].load(x + row[u] * K, col[u], K);
      else
        run[u].zero();
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (base + u * nwarps >= ntasks) break;  // warp-uniform
      const int64_t m = row[u], k = col[u];
      uint32_t key = run[u].max_key();
      if constexpr (GS == 128) {  // a group is four lanes' runs
        key = max(key, __shfl_xor_sync(0xffffffffu, key, 1));
        key = max(key, __shfl_xor_sync(0xffffffffu, key, 2));
      }
      const float amax = __uint_as_float(key);
      const int64_t g = k >> kShift;
      const bool scale_lane = (GS == 32 || (l & 3) == 0) && g < G;
      if (sfmt == 0) {
        const float s = scale_from_amax(amax, mx);
        if (scale_lane) reinterpret_cast<float *>(scales)[g * M + m] = s;
        run[u].template quant_store<F>(q + m * K, k, K, ScaleDiv(s));
      } else {
        // UE8M0: 2^e, e = ceil(log2(fl32(amax / MAX))); 1.0 for a zero group
        const int e = amax > 0.0f ? min(max(ceil_log2_pos(__fdiv_rn(amax, mx)), -127), 127) : 0;
        if (scale_lane) reinterpret_cast<uint8_t *>(scales)[g * M + m] = (uint8_t)(e + 127);
        run[u].template quant_store_pow2<F>(q + m * K, k, K, exp2_int(-e));
      }
    }
  }
}

// --------------------------------------------------- weight block 128x128 --
// One CTA per block: thread t covers row t/2, columns (t%2)*64 .. +64.
template <typename T>
__global__ void __launch_bounds__(256)
    quant_block_kernel(const T *__restrict__ w, int64_t N, int64_t K, int fmt, int sfmt,
                       uint8_t *__restrict__ q, void *scales) {
  __shared__ uint32_t red[8];
  __shared__ uint32_t amax_key;
  const float mx = fmt_max(fmt);
  const int64_t bn = blockIdx.y, bk = blockIdx.x, KB = (K + 127) / 128;
  const int t = threadIdx.x;
  const int64_t r = bn * 128 + (t >> 1);
  const int64_t cbase = bk * 128 + (t & 1) * 64;
  float v[64];
  uint32_t key = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t c = cbase + i * 8;
    float tmp[8];
    if (r < N && c < K) {
      Vec8<T>::load(w + r * K + c, tmp);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) tmp[j] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[i * 8 + j] = tmp[j];
      key = max(key, abs_key(tmp[j]));
    }
  }
  key = warp_max_u32(key);
  if (lane_id() == 0) red[t >> 5] = key;
  __syncthreads();
  if (t < 32) {
    uint32_t k2 = t < 8 ? red[t] : 0u;
    k2 = warp_max_u32(k2);
    if (t == 0) amax_key = k2;
  }
  __syncthreads();
  const float amax = __uint_as_float(amax_key);
  float s = scale_from_amax(amax, mx);
  uint8_t e8 = 127;
  if (sfmt == 1) {
    if (amax > 0.0f) {
      const int e = min(max(ceil_log2_pos(s), -127), 127);
      s = exp2_int(e);
      e8 = (uint8_t)(e + 127);
    } else {
      s = 1.0f;
    }
  }
  if (t == 0) {
    if (sfmt == 0)
      reinterpret_cast<float *>(scales)[bn * KB + bk] = s;
    else
      reinterpret_cast<uint8_t *>(scales)[bn * KB + bk] = e8;
  }
  const ScaleDiv d(s);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t c = cbase + i * 8;
    if (r < N && c < K) {
      float y[8];
      div8(d, v + i * 8, y);
      *reinterpret_cast<uint2 *>(q + r * K + c) = pack8(fmt, y);
    }
  }
}

// ------------------------------------------------------ two-level (MOSS) --
// One warp per (row, pair of 128-wide K slices); lane l holds elements
// [8l, 8l+8): the 1x32 block of lane l is l/4 (four lanes per block).
// Index of the packed local-factor word for (row r, slice g).
__device__ __forceinline__ int64_t mx_word_index(int64_t r, int64_t g, int64_t rpad) {
  return g * rpad + (r & ~(int64_t)127) + 4 * (r & 31) + ((r & 127) >> 5);
}

// kGlobal selects the global factor:
//   kMxTensor   two level (MOSS blog, section 4): S = fl32(tensor amax / MAX)
//               (= max_i fl32(amax_i / MAX)), one for the tensor;
//   kMxOneLevel plain MXFP8 (section 1): S = 1, each block's power of two the
//               smallest not below amax_i / MAX;
//   kMxRow      two level with a global factor per row: S_r = fl32(row amax /
//               MAX) from amax_in[r], written to global_out[r].
constexpr int kMxTensor = 0, kMxOneLevel = 1, kMxRow = 2;
// One warp per (row, 1024-wide window of K): lane l owns the 1x32 block
// 32w + l of the row (elements [32l, 32l + 32) of window w), so each lane
// forms one block's factor for its 32 elements; lanes 4c..4c+3 hold the four
// bytes of one packed word.  Rows are padded to a multiple of 128 (padding
// rows only write their words).  kU windows per warp at once, loads first.
template <typename T, int kGlobal, int F>
__global__ void __launch_bounds__(256, 3)
    quant_mx_kernel(const T *__restrict__ x, int64_t R, int64_t K,
                    const float *amax_in, float *global_out, uint8_t *__restrict__ q,
                    uint32_t *__restrict__ local) {
  constexpr bool kOneLevel = kGlobal == kMxOneLevel;
  constexpr int kU = sizeof(T) == 2 ? 2 : 1;
  const float mx = fmt_max(F);
  // two level: S == max_i fl32(amax_i / MAX)
  const float S_tensor = kGlobal == kMxTensor ? scale_from_amax(*amax_in, mx) : 1.0f;
  if (kGlobal != kMxRow && global_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *global_out = S_tensor;
  const int64_t G = K / 128, wins = (K + 1023) / 1024;
  const int64_t rpad = (R + 127) / 128 * 128, ntasks = rpad * wins;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const bool narrow = ntasks + kU * nwarps <= (int64_t)0xFFFFFFFFu;
  const uint32_t l = lane_id();
  for (int64_t base = warp; base < ntasks; base += kU * nwarps) {
    Run32<T> run[kU];
    int64_t row[kU], col[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t task = base + u * nwarps;
      int64_t w;
      split_task(task, wins, narrow, row[u], w);
      col[u] = w * 1024 + l * 32;
      if (task < ntasks && row[u] < R)
        run[u].load(x + row[u] * K, col[u], K);
      else
        run[u].zero();
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (base + u * nwarps >= ntasks) break;  // warp-uniform
      const int64_t r = row[u], k = col[u], g = k >> 7;
      const bool word_lane = (l & 3) == 0 && g < G;
      if (r >= R) {  // padding rows: factor 1 (byte 127)
        if (word_lane) local[mx_word_index(r, g, rpad)] = 0x7F7F7F7Fu;
        continue;
      }
      float S = S_tensor;
      if constexpr (kGlobal == kMxRow) {
        S = scale_from_amax(amax_in[r], mx);
        if (k == 0 && global_out != nullptr) global_out[r] = S;
      }
      const float amax_i = __uint_as_float(run[u].max_key());
      const float s_i = __fdiv_rn(amax_i, mx);     // step 1
      int e = 0;
      if (kOneLevel) {
        if (s_i > 0.0f) e = min(max(ceil_log2_pos(s_i), -127), 127);
      } else if (s_i > 0.0f) {
        const float ratio = __fdiv_rn(s_i, S);     // step 3
        e = ratio > 0.0f ? max(ceil_log2_pos(ratio), -127) : -127;
      }
      if (kOneLevel)
        run[u].template quant_store_pow2<F>(q + r * K, k, K, exp2_int(-e));
      else
        run[u].template quant_store<F>(q + r * K, k, K, ScaleDiv(S * exp2_int(e)));  // step 4: S * r_i
      // the four block bytes of a 128-wide slice into one word
      const uint32_t b = (uint32_t)(e + 127) & 0xFFu;
      const uint32_t b1 = __shfl_down_sync(0xffffffffu, b, 1);
      const uint32_t b2 = __shfl_down_sync(0xffffffffu, b, 2);
      const uint32_t b3 = __shfl_down_sync(0xffffffffu, b, 3);
      if (word_lane) local[mx_word_index(r, g, rpad)] = b | (b1 << 8) | (b2 << 16) | (b3 << 24);
    }
  }
}

// ------------------------------------------------- delayed-state update --
// One CTA: roll the history by -1, write the new amax at index 0, then take
// max(history) (NaN propagates, as a max over the array does) and update the
// scale when it is positive and finite.
// One amax-history step (the body of both launches): `old` is L floats of
// shared memory; every thread of the CTA takes part.
__device__ __forceinline__ void delayed_update_one(float *hist, float *scale,
                                                   const float *amax_cur, int64_t L, int fmt,
                                                   float *old) {
  __shared__ uint32_t red_key[32];
  __shared__ int red_nan[32];
  for (int64_t i = threadIdx.x; i < L; i += blockDim.x) old[i] = hist[i];
  __syncthreads();
  const float a = *amax_cur;
  uint32_t key = 0;
  int nan_seen = 0;
  for (int64_t i = threadIdx.x; i < L; i += blockDim.x) {
    const float v = (i == 0) ? a : old[(i + 1) % L];
    hist[i] = v;
    if (v != v) nan_seen = 1;
    // keys of non-negative floats order like uints; +inf is the largest
    else key = max(key, v > 0.0f ? __float_as_uint(v) : 0u);
  }
  key = warp_max_u32(key);
  nan_seen = __any_sync(0xffffffffu, nan_seen);
  if (lane_id() == 0) {
    red_key[threadIdx.x >> 5] = key;
    red_nan[threadIdx.x >> 5] = nan_seen;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int nw = (blockDim.x + 31) >> 5;
    uint32_t k = threadIdx.x < (uint32_t)nw ? red_key[threadIdx.x] : 0u;
    int nn = threadIdx.x < (uint32_t)nw ? red_nan[threadIdx.x] : 0;
    k = warp_max_u32(k);
    nn = __any_sync(0xffffffffu, nn);
    if (threadIdx.x == 0) {
      const float m = __uint_as_float(k);
      if (!nn && m > 0.0f && m <= 3.402823466e38f) *scale = __fdiv_rn(m, fmt_max(fmt));
    }
  }
}

__global__ void __launch_bounds__(1024)
    delayed_update_kernel(float *hist, float *scale, const float *amax_cur, int64_t L, int fmt) {
  extern __shared__ float old[];
  delayed_update_one(hist, scale, amax_cur, L, fmt, old);
}

// Several histories in one launch, one CTA each.
__global__ void __launch_bounds__(1024)
    delayed_update_multi_kernel(const __grid_constant__ DelayedItems items) {
  extern __shared__ float old[];
  const int b = (int)blockIdx.x;
  delayed_update_one(items.hist[b], items.scale[b], items.amax_cur[b], items.L[b], items.fmt[b],
                     old);
}

// ----------------------------------------------------------- launchers --
static int grid_for(int64_t work, int threads, int per_sm_blocks, int sms) {
  const int64_t need = (work + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * per_sm_blocks;
  return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

cudaError_t launch_amax(const void *x, int in_dt, int64_t n, float *out, int sms,
                        cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float), st);
  if (e != cudaSuccess || n == 0) return e;
  const int threads = 512, blocks = grid_for((n + 7) / 8, threads, 2, sms);
  if (in_dt == 0)
    amax_kernel<__nv_bfloat16><<<blocks, threads, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(x), n, reinterpret_cast<uint32_t *>(out));
  else
    amax_kernel<float><<<blocks, threads, 0, st>>>(static_cast<const float *>(x), n,
                                                    reinterpret_cast<uint32_t *>(out));
  return cudaGetLastError();
}

cudaError_t launch_quant_tensor(const void *x, int in_dt, int64_t rows, int64_t cols, int fmt,
                                const float *amax_in, const float *scale, float *scale_out,
                                uint8_t *q, uint8_t *qt, float *amax_out, int sms,
                                cudaStream_t st) {
  if (amax_out != nullptr) {
    cudaError_t e = cudaMemsetAsync(amax_out, 0, sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  uint32_t *ao = reinterpret_cast<uint32_t *>(amax_out);
  const bool fused = amax_out != nullptr;
  if (qt == nullptr) {
    const int64_t n = rows * cols;
    // one wave of resident CTAs (launch bounds: 3 per SM), a warp per
    // 1024-element window
    const int threads = 256, blocks = grid_for((n / 8 + 127) / 128 * 32, threads, 3, sms);
#define FP8K_QT(T, A)                                                                         \
  (fmt == 0 ? quant_tensor_kernel<T, 0, A><<<blocks, threads, 0, st>>>(                        \
                  static_cast<const T *>(x), n, amax_in, scale, scale_out, q, ao)              \
            : quant_tensor_kernel<T, 1, A><<<blocks, threads, 0, st>>>(                        \
                  static_cast<const T *>(x), n, amax_in, scale, scale_out, q, ao))
    if (in_dt == 0) {
      if (fused) FP8K_QT(__nv_bfloat16, true); else FP8K_QT(__nv_bfloat16, false);
    } else {
      if (fused) FP8K_QT(float, true); else FP8K_QT(float, false);
    }
#undef FP8K_QT
  } else {
    const int64_t ntiles = ((cols + kTT - 1) / kTT) * ((rows + kTT - 1) / kTT);
    const int64_t cap = (int64_t)sms * 2;
    const unsigned grid = (unsigned)(ntiles < cap ? ntiles : cap);
#define FP8K_QTT(T, A)                                                                        \
  (fmt == 0 ? quant_tensor_t_kernel<T, 0, A><<<grid, 256, 0, st>>>(                            \
                  static_cast<const T *>(x), rows, cols, amax_in, scale, scale_out, q, qt, ao) \
            : quant_tensor_t_kernel<T, 1, A><<<grid, 256, 0, st>>>(                            \
                  static_cast<const T *>(x), rows, cols, amax_in, scale, scale_out, q, qt, ao))
    if (in_dt == 0) {
      if (fused) FP8K_QTT(__nv_bfloat16, true); else FP8K_QTT(__nv_bfloat16, false);
    } else {
      if (fused) FP8K_QTT(float, true); else FP8K_QTT(float, false);
    }
#undef FP8K_QTT
  }
  return cudaGetLastError();
}

// A launch with programmatic stream serialization (the kernel calls
// grid_dependency_wait() before it touches memory).
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), int blocks, int threads, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename T, int GS>
static cudaError_t launch_group_kernel(const void *x, int64_t M, int64_t K, int fmt, int sfmt,
                                       uint8_t *q, void *scales, int sms, cudaStream_t st) {
  // one resident wave (launch bounds: 3 CTAs per SM)
  const int threads = 256, blocks = grid_for(M * ((K + 1023) / 1024) * 32, threads, 3, sms);
  const T *xt = static_cast<const T *>(x);
  if (fmt == 0) return launch_pdl(quant_group_kernel<T, 0, GS>, blocks, threads, st, xt, M, K, sfmt, q, scales);
  return launch_pdl(quant_group_kernel<T, 1, GS>, blocks, threads, st, xt, M, K, sfmt, q, scales);
}

cudaError_t launch_quant_group(const void *x, int in_dt, int64_t M, int64_t K, int fmt,
                               int sfmt, uint8_t *q, void *scales, int sms, cudaStream_t st) {
  if (in_dt == 0)
    return launch_group_kernel<__nv_bfloat16, 128>(x, M, K, fmt, sfmt, q, scales, sms, st);
  return launch_group_kernel<float, 128>(x, M, K, fmt, sfmt, q, scales, sms, st);
}

cudaError_t launch_quant_block(const void *w, int in_dt, int64_t N, int64_t K, int fmt,
                               int sfmt, uint8_t *q, void *scales, cudaStream_t st) {
  dim3 grid((unsigned)((K + 127) / 128), (unsigned)((N + 127) / 128));
  if (in_dt == 0)
    quant_block_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(w), N, K, fmt, sfmt, q, scales);
  else
    quant_block_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float *>(w), N, K, fmt,
                                                     sfmt, q, scales);
  return cudaGetLastError();
}

cudaError_t launch_quant_mx(const void *x, int in_dt, int64_t R, int64_t K, int fmt,
                            const float *amax, float *global_out, uint8_t *q, uint32_t *local,
                            int sms, cudaStream_t st, bool per_row) {
  const int64_t rpad = (R + 127) / 128 * 128;
  const int threads = 256, blocks = grid_for(rpad * ((K + 1023) / 1024) * 32, threads, 3, sms);
  const int kind = amax == nullptr ? kMxOneLevel : (per_row ? kMxRow : kMxTensor);
#define FP8K_QMX(T, G)                                                                         \
  (fmt == 0 ? quant_mx_kernel<T, G, 0><<<blocks, threads, 0, st>>>(                            \
                  static_cast<const T *>(x), R, K, amax, global_out, q, local)                 \
            : quant_mx_kernel<T, G, 1><<<blocks, threads, 0, st>>>(                            \
                  static_cast<const T *>(x), R, K, amax, global_out, q, local))
  if (in_dt == 0) {
    if (kind == kMxTensor) FP8K_QMX(__nv_bfloat16, kMxTensor);
    else if (kind == kMxOneLevel) FP8K_QMX(__nv_bfloat16, kMxOneLevel);
    else FP8K_QMX(__nv_bfloat16, kMxRow);
  } else {
    if (kind == kMxTensor) FP8K_QMX(float, kMxTensor);
    else if (kind == kMxOneLevel) FP8K_QMX(float, kMxOneLevel);
    else FP8K_QMX(float, kMxRow);
  }
#undef FP8K_QMX
  return cudaGetLastError();
}

// ------------------------------------------------- weight block 32 x 32 --
// (32, 32) weight blocks with UE8M0 scales (Transformers fine-grained FP8,
// 八: a non-default weight_block_size; 七: UE8M0 rounded up, quantize with
// it).  One warp per block: lane l holds row n0 + l of the block.  Writes the
// codes, the block bytes [ceil(N/32), K/32] (nullable) and, for every row,
// the block byte of each 1x32 piece into the packed E8M0 word layout of the
// two-level GEMM (rows past N up to R_pad get byte 127), so fp8_gemm_mx
// contracts these weights with one-level MXFP8 activations directly.
// kF32: fp32 scales fl32(amax / MAX) (1.0 for an all-zero block) written to
// scales_f32 [ceil(N/32), K/32], each block divided by its own scale; no MX
// words (the per-32 FP32 GEMM promotes them on the CUDA cores).
template <typename T, int F, bool kF32>
__global__ void __launch_bounds__(256)
    quant_block32_kernel(const T *__restrict__ w, int64_t N, int64_t K,
                         uint8_t *__restrict__ q, uint8_t *__restrict__ scales,
                         uint32_t *__restrict__ local, float *__restrict__ scales_f32) {
  const float mx = fmt_max(F);
  const int64_t KB = K / 32, rpad = kF32 ? (N + 31) / 32 * 32 : (N + 127) / 128 * 128;
  const int64_t nblk = (rpad / 32) * KB;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t l = lane_id();
  uint8_t *local8 = reinterpret_cast<uint8_t *>(local);
  for (int64_t b = warp; b < nblk; b += nwarps) {
    const int64_t bn = b / KB, bk = b % KB;
    const int64_t n = bn * 32 + l, k0 = bk * 32;
    const bool valid = n < N;
    Raw8<T> raw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (valid)
        raw[i].load_stream(w + n * K + k0 + 8 * i);
      else
        raw[i].zero();
    }
    uint32_t key_a = 0, key_b = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) raw[i].max_abs(key_a, key_b);
    const uint32_t key = warp_max_u32(Raw8<T>::merge_keys(key_a, key_b));
    const float amax = __uint_as_float(key);
    if constexpr (kF32) {
      const float sc = scale_from_amax(amax, mx);
      if (l == 0) scales_f32[bn * KB + bk] = sc;
      if (valid) {
        const ScaleDiv d(sc);
        uint2 c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = quant8_block<F>(raw[i], d);
        uint4 *dst = reinterpret_cast<uint4 *>(q + n * K + k0);
        dst[0] = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
        dst[1] = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
      }
      continue;
    }
    int e = 0;
    if (amax > 0.0f) e = min(max(ceil_log2_pos(__fdiv_rn(amax, mx)), -127), 127);
    const uint8_t byte = (uint8_t)(e + 127);
    if (l == 0 && scales != nullptr && bn * 32 < N) scales[bn * KB + bk] = byte;
    // this row's byte in the packed word of (row n, 128-wide slice k0 / 128)
    local8[4 * mx_word_index(n, k0 / 128, rpad) + (k0 % 128) / 32] = valid ? byte : (uint8_t)127;
    if (valid) {
      const uint64_t inv2 = f32x2_pack(exp2_int(-e), exp2_int(-e));
      uint2 c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] = quant8_pow2<F>(raw[i], inv2);
      uint4 *dst = reinterpret_cast<uint4 *>(q + n * K + k0);
      dst[0] = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
      dst[1] = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
    }
  }
}

cudaError_t launch_quant_block32(const void *w, int in_dt, int64_t N, int64_t K, int fmt,
                                 uint8_t *q, uint8_t *scales, uint32_t *local, int sms,
                                 cudaStream_t st) {
  const int64_t rpad = (N + 127) / 128 * 128;
  const int threads = 256, blocks = grid_for((rpad / 32) * (K / 32) * 32, threads, 8, sms);
#define FP8K_QB32(T, F)                                                                       \
  quant_block32_kernel<T, F, false><<<blocks, threads, 0, st>>>(static_cast<const T *>(w), N, K, \
                                                                q, scales, local, nullptr)
  if (in_dt == 0) {
    if (fmt == 0) FP8K_QB32(__nv_bfloat16, 0); else FP8K_QB32(__nv_bfloat16, 1);
  } else {
    if (fmt == 0) FP8K_QB32(float, 0); else FP8K_QB32(float, 1);
  }
#undef FP8K_QB32
  return cudaGetLastError();
}

cudaError_t launch_quant_block32_f32(const void *w, int in_dt, int64_t N, int64_t K, int fmt,
                                     uint8_t *q, float *scales, int sms, cudaStream_t st) {
  const int64_t npad = (N + 31) / 32 * 32;
  const int threads = 256, blocks = grid_for((npad / 32) * (K / 32) * 32, threads, 8, sms);
#define FP8K_QB32F(T, F)                                                                     \
  quant_block32_kernel<T, F, true><<<blocks, threads, 0, st>>>(static_cast<const T *>(w), N, K, \
                                                               q, nullptr, nullptr, scales)
  if (in_dt == 0) {
    if (fmt == 0) FP8K_QB32F(__nv_bfloat16, 0); else FP8K_QB32F(__nv_bfloat16, 1);
  } else {
    if (fmt == 0) FP8K_QB32F(float, 0); else FP8K_QB32F(float, 1);
  }
#undef FP8K_QB32F
  return cudaGetLastError();
}

cudaError_t launch_quant_group32(const void *x, int in_dt, int64_t M, int64_t K, int fmt,
                                 int sfmt, uint8_t *q, void *scales, int sms, cudaStream_t st) {
  if (in_dt == 0)
    return launch_group_kernel<__nv_bfloat16, 32>(x, M, K, fmt, sfmt, q, scales, sms, st);
  return launch_group_kernel<float, 32>(x, M, K, fmt, sfmt, q, scales, sms, st);
}

// ------------------------------------------ UE8M0 group scales -> MX words --
// The per-K-group GEMM with UE8M0 scales runs as the block-scaled GEMM: each
// 1x128 activation scale and 128x128 weight-block scale becomes the four
// equal E8M0 bytes of its row's packed word for that 128-wide K slice (the
// tensor core then applies the same factor to each 1x32 sub-block, which is
// the group's factor).  Word i of slice g (i < R_pad) belongs to row
// (i & ~127) + 32 (i & 3) + ((i & 127) >> 2), the inverse of mx_word_index;
// padding rows get byte 127 (factor 1).
// Grid: x over the words of one K slice (4 per thread), y over the K slices
// g, z = operand (0 A, 1 B); no divisions.
__global__ void __launch_bounds__(256)
    ue8m0_words_kernel(const uint8_t *__restrict__ sa, const uint8_t *__restrict__ sb,
                       int64_t M, int64_t N, int64_t G, uint32_t *__restrict__ la,
                       uint32_t *__restrict__ lb) {
  const bool is_a = blockIdx.z == 0;
  const int64_t R = is_a ? M : N, pad = (R + 127) / 128 * 128;
  for (int64_t g = blockIdx.y; g < G; g += gridDim.y) {
    uint32_t *dst = (is_a ? la : lb) + g * pad;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t w = ((int64_t)blockIdx.x * 4 + u) * blockDim.x + threadIdx.x;
      if (w >= pad) break;
      const int64_t r = (w & ~(int64_t)127) + 32 * (w & 3) + ((w & 127) >> 2);
      uint32_t b = 127u;
      if (r < R) b = is_a ? sa[g * M + r] : sb[(r >> 7) * G + g];
      dst[w] = b * 0x01010101u;
    }
  }
}

cudaError_t launch_ue8m0_words(const uint8_t *sa, const uint8_t *sb, int64_t M, int64_t N,
                               int64_t K, uint32_t *la, uint32_t *lb, int sms, cudaStream_t st) {
  (void)sms;
  const int64_t G = K / 128, pad = ((M > N ? M : N) + 127) / 128 * 128;
  const dim3 grid((unsigned)((pad + 1023) / 1024), (unsigned)(G < 65535 ? G : 65535), 2);
  ue8m0_words_kernel<<<grid, 256, 0, st>>>(sa, sb, M, N, G, la, lb);
  return cudaGetLastError();
}

// Expert-grouped rows (expert e owns rows [o_e, o_{e+1}), cut into
// ceil(rows_e / 128) row tiles, the tiles of all experts in order): the A
// words are stored per row tile, [tile][K/128][128] in the MMA's order, so a
// tile that starts at any row reads one contiguous 512-byte slice per k
// block.  The B words use the plain layout over the E * N weight rows
// (N % 128 == 0, so no expert's rows share a 128-row block).
__global__ void __launch_bounds__(256)
    ue8m0_words_experts_kernel(const uint8_t *__restrict__ sa, const uint8_t *__restrict__ sb,
                               const int32_t *__restrict__ offsets, int E, int64_t M, int64_t N,
                               int64_t G, int64_t tmax, uint32_t *__restrict__ la,
                               uint32_t *__restrict__ lb) {
  __shared__ int32_t rt0[kMaxExperts + 1];   // first row tile of each expert
  __shared__ int32_t row0[kMaxExperts + 1];  // first row of each expert
  if (threadIdx.x < 32) {
    const int l = (int)threadIdx.x;
    int cnt[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = 8 * l + i;
      cnt[i] = 0;
      if (e < E) {
        const int32_t r0 = offsets[e], r1 = offsets[e + 1];
        row0[e] = r0;
        cnt[i] = r1 > r0 ? (r1 - r0 + 127) / 128 : 0;
        if (e == E - 1) row0[E] = r1;
      }
      sum += cnt[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (l >= o) incl += v;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = 8 * l + i;
      if (e < E) rt0[e] = run;
      run += cnt[i];
      if (e == E - 1) rt0[E] = run;
    }
  }
  __syncthreads();
  // grid: y over the K slices g, z = operand (0 A, 1 B), x over a slice's words
  const int T = rt0[E];
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t g = blockIdx.y; g < G; g += gridDim.y) {
    if (blockIdx.z == 0) {
      // A: word p of row tile j at la[(j * G + g) * 128 + p]
      for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < tmax * 128; w += stride) {
        const int64_t j = w >> 7, p = w & 127;
        const int64_t ir = 32 * (p & 3) + (p >> 2);  // tile row of word p
        uint32_t b = 127u;
        if (j < T) {
          int lo = 0, hi = E;  // the expert with rt0[lo] <= j < rt0[lo + 1]
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (rt0[mid] <= j) lo = mid; else hi = mid;
          }
          while (lo + 1 < E && rt0[lo + 1] <= j) ++lo;
          const int64_t r = row0[lo] + (j - rt0[lo]) * 128 + ir;
          if (r < row0[lo + 1]) b = sa[g * M + r];
        }
        la[(j * G + g) * 128 + p] = b * 0x01010101u;
      }
    } else {
      // B: the plain layout over the E * N weight rows (e = r / N, 32-bit)
      const int64_t R = (int64_t)E * N;
      const uint32_t n32 = (uint32_t)N;
      for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < R; w += stride) {
        const int64_t r = (w & ~(int64_t)127) + 32 * (w & 3) + ((w & 127) >> 2);
        const uint32_t e = (uint32_t)r / n32, n = (uint32_t)r - e * n32;
        const uint32_t b = sb[(int64_t)e * ((N / 128) * G) + (int64_t)(n >> 7) * G + g];
        lb[g * R + w] = b * 0x01010101u;
      }
    }
  }
}

cudaError_t launch_ue8m0_words_experts(const uint8_t *sa, const uint8_t *sb,
                                       const int32_t *offsets, int E, int64_t M, int64_t N,
                                       int64_t K, int64_t tmax, uint32_t *la, uint32_t *lb,
                                       int sms, cudaStream_t st) {
  (void)sms;
  const int64_t G = K / 128;
  const int64_t per_slice = tmax * 128 > (int64_t)E * N ? tmax * 128 : (int64_t)E * N;
  const int64_t bx = (per_slice + 4 * 256 - 1) / (4 * 256);
  const dim3 grid((unsigned)bx, (unsigned)(G < 65535 ? G : 65535), 2);
  ue8m0_words_experts_kernel<<<grid, 256, 0, st>>>(sa, sb, offsets, E, M, N, G, tmax, la, lb);
  return cudaGetLastError();
}

// ------------------------------------------------------------- row amax --
// amax_out[r] = max |x[r, :]|: one warp per row, 16-byte loads, the same
// order-preserving keys as the tensor amax (exact).
template <typename T>
__global__ void __launch_bounds__(256)
    row_amax_kernel(const T *__restrict__ x, int64_t R, int64_t K, float *__restrict__ out) {
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t l = lane_id();
  for (int64_t r = warp; r < R; r += nwarps) {
    uint32_t key_a = 0, key_b = 0;
    const T *row = x + r * K;
    for (int64_t v = l; v < K / 8; v += 32) {
      Raw8<T> raw;
      raw.load_stream(row + v * 8);
      raw.max_abs(key_a, key_b);
    }
    uint32_t key = Raw8<T>::merge_keys(key_a, key_b);
    for (int64_t i = K / 8 * 8 + l; i < K; i += 32) key = max(key, abs_key(load1(row + i)));
    key = warp_max_u32(key);
    if (l == 0) out[r] = __uint_as_float(key);
  }
}

cudaError_t launch_row_amax(const void *x, int in_dt, int64_t R, int64_t K, float *out, int sms,
                            cudaStream_t st) {
  const int threads = 256, blocks = grid_for(R * 32, threads, 8, sms);
  if (in_dt == 0)
    row_amax_kernel<__nv_bfloat16><<<blocks, threads, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(x), R, K, out);
  else
    row_amax_kernel<float><<<blocks, threads, 0, st>>>(static_cast<const float *>(x), R, K, out);
  return cudaGetLastError();
}

// ------------------------------------------------- block dequantization --
// out[n, k] = decode(q[n, k]) * scale of block (n/128, k/128), rounded to bf16
// (Transformers fine-grained FP8, 五).  Eight codes per thread: the FP8 -> f16
// conversion is exact for both formats, the product is formed in fp32.
__global__ void __launch_bounds__(256)
    dequant_block_kernel(const uint8_t *__restrict__ q, int64_t N, int64_t K, int fmt,
                         int sfmt, const void *scales, __nv_bfloat16 *__restrict__ out) {
  const int64_t KB = (K + 127) / 128;
  const int64_t nvec = N * K / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    const int64_t e0 = i * 8, n = e0 / K, k = e0 % K;
    const int64_t bi = (n >> 7) * KB + (k >> 7);
    const float sc = sfmt == 0 ? static_cast<const float *>(scales)[bi]
                               : exp2_int((int)static_cast<const uint8_t *>(scales)[bi] - 127);
    const uint2 c = __ldcs(reinterpret_cast<const uint2 *>(q) + i);
    const uint32_t w[2] = {c.x, c.y};
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint16_t pair = (uint16_t)(w[h >> 1] >> (16 * (h & 1)));
      uint32_t f16x2;
      if (fmt == 0)
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f16x2) : "h"(pair));
      else
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(f16x2) : "h"(pair));
      const __half2 hv = *reinterpret_cast<const __half2 *>(&f16x2);
      const float lo = __low2float(hv) * sc, hi = __high2float(hv) * sc;
      __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
      o[h] = *reinterpret_cast<uint32_t *>(&b);
    }
    __stcs(reinterpret_cast<uint4 *>(out) + i, make_uint4(o[0], o[1], o[2], o[3]));
  }
}

cudaError_t launch_dequant_block(const uint8_t *q, int64_t N, int64_t K, int fmt, int sfmt,
                                 const void *scales, void *out, int sms, cudaStream_t st) {
  const int64_t nvec = N * K / 8;
  const int threads = 256, blocks = grid_for(nvec, threads, 8, sms);
  dequant_block_kernel<<<blocks, threads, 0, st>>>(q, N, K, fmt, sfmt, scales,
                                                   static_cast<__nv_bfloat16 *>(out));
  return cudaGetLastError();
}

// MOSS automatic weight scaling (eq. 10): scale = (amax_0 + eta * t) / MAX,
// with eta * t rounded to fp32 on the host; one thread, no reads of the weight.
__global__ void auto_scale_kernel(const float *amax0, float grow, int fmt, float *scale) {
  if (threadIdx.x == 0) *scale = __fdiv_rn(__fadd_rn(*amax0, grow), fmt_max(fmt));
}

cudaError_t launch_auto_scale(const float *amax0, double grow, int fmt, float *scale,
                              cudaStream_t st) {
  auto_scale_kernel<<<1, 32, 0, st>>>(amax0, (float)grow, fmt, scale);
  return cudaGetLastError();
}

cudaError_t launch_delayed_update(float *hist, float *scale, const float *amax_cur, int64_t L,
                                  int fmt, cudaStream_t st) {
  const size_t smem = (size_t)L * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(delayed_update_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  delayed_update_kernel<<<1, 1024, smem, st>>>(hist, scale, amax_cur, L, fmt);
  return cudaGetLastError();
}

cudaError_t launch_delayed_update_multi(const DelayedItems &items, cudaStream_t st) {
  if (items.count < 1 || items.count > kMaxDelayed) return cudaErrorInvalidValue;
  int64_t lmax = 1;
  for (int i = 0; i < items.count; ++i) lmax = items.L[i] > lmax ? items.L[i] : lmax;
  const size_t smem = (size_t)lmax * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(delayed_update_multi_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  delayed_update_multi_kernel<<<items.count, 1024, smem, st>>>(items);
  return cudaGetLastError();
}

}  // namespace fp8k
