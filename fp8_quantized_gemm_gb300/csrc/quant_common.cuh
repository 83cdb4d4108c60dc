// Element access shared by the quantization kernels: 16-byte vector loads of
// bf16 / fp32 inputs, the |x| key reduction, the packed FP8 store, and the
// block-wide max.
#pragma once

#include "common.cuh"

namespace fp8k {

// ---------------------------------------------------------------- loads --
// Eight consecutive input elements as fp32 (bf16: one 16-byte load; f32: two).
template <typename T>
struct Vec8;

template <>
struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ void load_stream(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

template <>
struct Vec8<float> {
  static __device__ __forceinline__ void load(const float *p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  static __device__ __forceinline__ void load_stream(const float *p, float (&v)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// Raw 16-byte vectors holding 8 elements (bf16: one uint4; f32: two), kept
// undecoded in registers until used.
template <typename T>
struct Raw8 {
  static constexpr int kWords = sizeof(T) * 8 / 16;
  uint4 w[kWords];
  __device__ __forceinline__ void load_stream(const T *p) {
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = __ldcs(reinterpret_cast<const uint4 *>(p) + i);
  }
  // from shared memory (16-byte aligned)
  __device__ __forceinline__ void load_shared(const uint8_t *p) {
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = reinterpret_cast<const uint4 *>(p)[i];
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  // Running max of |x| over the 8 elements as order-preserving keys.  bf16:
  // key_a holds two 16-bit keys (|x| bits of the even and odd elements, max
  // taken per halfword), so one mask and one paired max per element pair;
  // merge_keys folds them into the fp32 bit pattern of |x|.  fp32: two
  // running uint32 keys.
  __device__ __forceinline__ void max_abs(uint32_t &key_a, uint32_t &key_b) const {
    if constexpr (sizeof(T) == 2) {
      (void)key_b;
#pragma unroll
      for (int i = 0; i < kWords; ++i) {
        const uint32_t u[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) key_a = __vmaxu2(key_a, u[j] & 0x7FFF7FFFu);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kWords; ++i) {
        key_a = max(key_a, w[i].x & 0x7FFFFFFFu);
        key_b = max(key_b, w[i].y & 0x7FFFFFFFu);
        key_a = max(key_a, w[i].z & 0x7FFFFFFFu);
        key_b = max(key_b, w[i].w & 0x7FFFFFFFu);
      }
    }
  }
  // The eight elements' sign bits at the sign bits of their eight packed
  // FP8 codes (sign-magnitude: bit 7 of each code byte).
  __device__ __forceinline__ uint2 code_signs() const {
    if constexpr (sizeof(T) == 2) {
      // bf16 element 2i sits in bits 0-15 of a word, 2i+1 in bits 16-31: the
      // sign bytes are bytes 1 and 3 of each word
      return make_uint2(__byte_perm(w[0].x, w[0].y, 0x7531) & 0x80808080u,
                        __byte_perm(w[0].z, w[0].w, 0x7531) & 0x80808080u);
    } else {
      auto s4 = [](const uint4 &v) {
        return __byte_perm(__byte_perm(v.x, v.y, 0x0073), __byte_perm(v.z, v.w, 0x7300),
                           0x7610) & 0x80808080u;
      };
      return make_uint2(s4(w[0]), s4(w[1]));
    }
  }
  // Combine the two running keys of max_abs into one fp32 |x| key.
  static __device__ __forceinline__ uint32_t merge_keys(uint32_t key_a, uint32_t key_b) {
    if constexpr (sizeof(T) == 2) return max(key_a & 0xFFFF0000u, key_a << 16);
    return max(key_a, key_b);
  }
  __device__ __forceinline__ void decode(float (&v)[8]) const {
    if constexpr (sizeof(T) == 2) {
      const uint32_t u[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(u[i] << 16);
        v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        v[4 * i] = __uint_as_float(w[i].x);
        v[4 * i + 1] = __uint_as_float(w[i].y);
        v[4 * i + 2] = __uint_as_float(w[i].z);
        v[4 * i + 3] = __uint_as_float(w[i].w);
      }
    }
  }
};

template <typename T>
__device__ __forceinline__ float load1(const T *p);
template <>
__device__ __forceinline__ float load1<__nv_bfloat16>(const __nv_bfloat16 *p) {
  return __bfloat162float(*p);
}
template <>
__device__ __forceinline__ float load1<float>(const float *p) { return *p; }

// Two values -> two codes of the format F (0 E4M3, 1 E5M2), fixed at compile
// time so that the hot loops issue one conversion per pair.
template <int F>
__device__ __forceinline__ uint32_t cvt8x2(float lo, float hi) {
  if constexpr (F == 0)
    return cvt_e4m3x2(lo, hi);
  else
    return cvt_e5m2x2(lo, hi);
}

// 8 values -> 8 codes packed little-endian into a uint2.
template <int F>
__device__ __forceinline__ uint2 pack8(const float (&y)[8]) {
  const uint32_t c0 = cvt8x2<F>(y[0], y[1]), c1 = cvt8x2<F>(y[2], y[3]);
  const uint32_t c2 = cvt8x2<F>(y[4], y[5]), c3 = cvt8x2<F>(y[6], y[7]);
  return make_uint2(__byte_perm(c0, c1, 0x5410), __byte_perm(c2, c3, 0x5410));
}
// the same with the format chosen at run time (cold paths)
__device__ __forceinline__ uint2 pack8(int fmt, const float (&y)[8]) {
  return fmt == 0 ? pack8<0>(y) : pack8<1>(y);
}

// ---------------------------------------------- packed bf16 vectors --
// Eight bf16 values held as a 16-byte vector of packed pairs (element 2i in
// the low half of word i), quantized on a scale's fast path (ScaleDiv::fast)
// with fewer instructions than decoding them and dividing signed values:
//   - the running max of |x| is taken on the 16-bit halves (key2 holds two
//     16-bit keys; bf16_key_merge folds them into the fp32 bits of |x|);
//   - the quotient is formed from |x| clamped to ScaleDiv::bound (min.NaN:
//     a NaN stays NaN), so the bounded quotient cannot overflow and every
//     clamped value still saturates;
//   - the sign is put back from the bf16 sign bits into the codes' bit 7
//     (a NaN code keeps its input's sign).
// The codes equal those of dividing the signed values (div_by_scale).
__device__ __forceinline__ float min_nan_abs(float x, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(fabsf(x)), "f"(b));
  return r;
}

__device__ __forceinline__ void bf16x8_quotients(const uint4 w, const ScaleDiv &d, uint32_t &key2,
                                                 float (&y)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
  float x[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    key2 = __vmaxu2(key2, u[i] & 0x7FFF7FFFu);
    x[2 * i] = min_nan_abs(__uint_as_float(u[i] << 16), d.bound);
    x[2 * i + 1] = min_nan_abs(__uint_as_float(u[i] & 0xFFFF0000u), d.bound);
  }
#pragma unroll
  for (int j = 0; j < 8; j += 2) div_by_scale2_bounded(x[j], x[j + 1], d.ns2, d.y2, y[j], y[j + 1]);
}

// codes of non-negative quotients with the signs of the bf16 words put back
__device__ __forceinline__ uint2 bf16x8_with_signs(const uint2 c, const uint4 w) {
  return make_uint2(c.x | (__byte_perm(w.x, w.y, 0x7531) & 0x80808080u),
                    c.y | (__byte_perm(w.z, w.w, 0x7531) & 0x80808080u));
}

template <int F>
__device__ __forceinline__ uint2 quant_bf16x8(const uint4 w, const ScaleDiv &d, uint32_t &key2) {
  float y[8];
  bf16x8_quotients(w, d, key2, y);
  return bf16x8_with_signs(pack8<F>(y), w);
}

// the two 16-bit |x| keys of key2 as one fp32 |x| key
__device__ __forceinline__ uint32_t bf16_key_merge(uint32_t key2) {
  return max(key2 & 0xFFFF0000u, key2 << 16);
}

// Eight quotients v[j] / s by one scale (ScaleDiv; the fast/slow choice is
// per scale, so it diverges only between groups with extreme scales).
__device__ __forceinline__ void div8(const ScaleDiv &d, const float *v, float (&y)[8]) {
  const float(&v8)[8] = *reinterpret_cast<const float(*)[8]>(v);
  if (d.fast)
    d.div8<true>(v8, y);
  else
    d.div8<false>(v8, y);
}

// Block-wide max of a uint32 key, then one atomicMax per block.
__device__ __forceinline__ void block_max_to(uint32_t key, uint32_t *dst) {
  __shared__ uint32_t red[32];
  key = warp_max_u32(key);
  const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  if (lane_id() == 0) red[w] = key;
  __syncthreads();
  if (w == 0) {
    uint32_t k = lane_id() < (uint32_t)nw ? red[lane_id()] : 0u;
    k = warp_max_u32(k);
    if (lane_id() == 0 && k != 0u) atomicMax(dst, k);
  }
}

// Codes of the eight elements of r divided by d.s, for a scale formed from
// this tensor's own amax (d.fast checked by the caller): the bounded packed
// quotient, the saturating cast, then each element's sign put into its code
// (a zero or underflowed quotient becomes +-0 with the sign of x, as the
// IEEE quotient would).
template <int F, typename T>
__device__ __forceinline__ uint2 quant8_own_scale(const Raw8<T> &r, const ScaleDiv &d) {
  float x[8], y[8];
  r.decode(x);
#pragma unroll
  for (int j = 0; j < 8; j += 2) div_by_scale2_bounded(x[j], x[j + 1], d.ns2, d.y2, y[j], y[j + 1]);
  const uint2 c = pack8<F>(y);
  const uint2 sg = r.code_signs();
  return make_uint2(c.x | sg.x, c.y | sg.y);
}

// The same codes through IEEE division (scales outside the fast range).
template <int F, typename T>
__device__ __forceinline__ uint2 quant8_ieee(const Raw8<T> &r, const ScaleDiv &d) {
  float x[8], y[8];
  r.decode(x);
  d.div8<false>(x, y);
  return pack8<F>(y);
}

// Codes of eight elements divided by a power-of-two scale s = 2^e, given as
// the packed pair {2^-e, 2^-e}: the reciprocal of a power of two is exact,
// so x * 2^-e rounds the same real number as x / s, once.
template <int F, typename T>
__device__ __forceinline__ uint2 quant8_pow2(const Raw8<T> &r, uint64_t inv2) {
  float x[8], y[8];
  r.decode(x);
#pragma unroll
  for (int j = 0; j < 8; j += 2) f32x2_unpack(f32x2_mul(f32x2_pack(x[j], x[j + 1]), inv2), y[j], y[j + 1]);
  return pack8<F>(y);
}

// A lane's run of 32 consecutive elements of one row (four Raw8 vectors),
// for the kernels where each lane owns whole scale blocks (1x32) or a
// quarter of one (1x128).  Vectors at or past the row's end K read as zero
// and are not stored (K % 16 == 0, so each 16-element half is whole).
template <typename T>
struct Run32 {
  Raw8<T> v[4];
  __device__ __forceinline__ void load(const T *row, int64_t k, int64_t K) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (k + 8 * i < K)
        v[i].load_stream(row + k + 8 * i);
      else
        v[i].zero();
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i].zero();
  }
  // max |x| of the 32 elements as an fp32 bit pattern
  __device__ __forceinline__ uint32_t max_key() const {
    uint32_t key_a = 0, key_b = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i].max_abs(key_a, key_b);
    return Raw8<T>::merge_keys(key_a, key_b);
  }
  // codes of the 32 elements divided by the power-of-two scale 1 / inv
  // (inv = 2^-e exactly, so the product is the correctly rounded quotient),
  // stored at row_q + k
  template <int F>
  __device__ __forceinline__ void quant_store_pow2(uint8_t *row_q, int64_t k, int64_t K,
                                                   float inv) const {
    const uint64_t inv2 = f32x2_pack(inv, inv);
    uint2 c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = quant8_pow2<F>(v[i], inv2);
    if (k < K) *reinterpret_cast<uint4 *>(row_q + k) = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
    if (k + 16 < K)
      *reinterpret_cast<uint4 *>(row_q + k + 16) = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
  }
  // codes of the 32 elements divided by d.s (a scale formed from an amax
  // that covers them), stored at row_q + k
  template <int F>
  __device__ __forceinline__ void quant_store(uint8_t *row_q, int64_t k, int64_t K,
                                              const ScaleDiv &d) const {
    uint2 c[4];
    if (d.fast) {
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] = quant8_own_scale<F>(v[i], d);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] = quant8_ieee<F>(v[i], d);
    }
    if (k < K) *reinterpret_cast<uint4 *>(row_q + k) = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
    if (k + 16 < K)
      *reinterpret_cast<uint4 *>(row_q + k + 16) = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
  }
};

// Codes of eight elements divided by a scale formed from the amax of a block
// that contains them (so |x / s| stays within the format's range): the packed
// bounded quotient when the scale is in the fast range, IEEE division
// otherwise (tiny or huge scales; a NaN amax).
template <int F, typename T>
__device__ __forceinline__ uint2 quant8_block(const Raw8<T> &r, const ScaleDiv &d) {
  return d.fast ? quant8_own_scale<F>(r, d) : quant8_ieee<F>(r, d);
}

// task -> (row, column task) of a row-major task space with `per_row` tasks
// per row; `narrow` (the whole space below 2^32) takes the 32-bit division.
__device__ __forceinline__ void split_task(int64_t task, int64_t per_row, bool narrow,
                                           int64_t &row, int64_t &col) {
  if (narrow) {
    const uint32_t t = (uint32_t)task, d = (uint32_t)per_row, r = t / d;
    row = r;
    col = t - r * d;
  } else {
    row = task / per_row;
    col = task - row * per_row;
  }
}

}  // namespace fp8k
