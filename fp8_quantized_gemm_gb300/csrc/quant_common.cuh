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

// 8 values -> 8 codes packed little-endian into a uint2.
__device__ __forceinline__ uint2 pack8(int fmt, const float (&y)[8]) {
  const uint32_t c0 = cvt_fp8x2(fmt, y[0], y[1]), c1 = cvt_fp8x2(fmt, y[2], y[3]);
  const uint32_t c2 = cvt_fp8x2(fmt, y[4], y[5]), c3 = cvt_fp8x2(fmt, y[6], y[7]);
  return make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
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
template <typename T>
__device__ __forceinline__ uint2 quant8_own_scale(const Raw8<T> &r, int fmt, const ScaleDiv &d) {
  float x[8], y[8];
  r.decode(x);
#pragma unroll
  for (int j = 0; j < 8; j += 2) div_by_scale2_bounded(x[j], x[j + 1], d.ns2, d.y2, y[j], y[j + 1]);
  const uint2 c = pack8(fmt, y);
  const uint2 sg = r.code_signs();
  return make_uint2(c.x | sg.x, c.y | sg.y);
}

// The same codes through IEEE division (scales outside the fast range).
template <typename T>
__device__ __forceinline__ uint2 quant8_ieee(const Raw8<T> &r, int fmt, const ScaleDiv &d) {
  float x[8], y[8];
  r.decode(x);
  d.div8<false>(x, y);
  return pack8(fmt, y);
}

}  // namespace fp8k
