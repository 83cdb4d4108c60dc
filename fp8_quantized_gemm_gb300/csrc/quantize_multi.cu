// Current scaling of several tensors in ONE persistent launch: for every
// tensor t, amax_t = max |x_t|, s_t = fl32(amax_t / MAX) (1.0 for amax 0) and
// q_t = RNE_fp8(clip(x_t / s_t)) -- the Flax guide's current scaling
// (section 2.2), the same bytes as fp8_amax followed by fp8_quantize_tensor.
//
// The two passes over every tensor (reduce, then quantize) are pipelined
// across the tensors inside one cooperative grid, one CTA per SM:
//
//   warp 0      bulk-copies (cp.async.bulk) the CTA's share of tensor 0, 1, ...
//               into ring A: the amax stream, HBM-bound;
//   warp 1      the same shares again into ring B: the quantize stream (mostly
//               L2 hits: the tensor was read by the amax pass just before);
//   warps 2-13  reduce ring A; after its last chunk of tensor t the CTA
//               publishes its max (atomicMax on a key) and counts itself in;
//   warps 14-29 quantize ring B: before tensor t they wait until every CTA has
//               counted in for t (a bounded spin on the counter), then divide
//               by s_t, cast on store.  s_t comes from this tensor's own amax,
//               so every quotient is finite and at most MAX (1 + 2^-23): the
//               unguarded packed quotient applies (quant8_own_scale).
//
// So while the quantize warps run the ALU-heavy pass over tensor t, the amax
// warps are already streaming tensor t+1 from HBM.  Chunks are 24 KB of input
// (a multiple of 16 bytes, as the bulk copy needs); CTA b takes chunks b,
// b + G, ... of every tensor.  Elements past the last full 8-element vector
// are handled by CTA 0 with scalar accesses.
#include "common.cuh"
#include "kernels.h"
#include "quant_common.cuh"

namespace fp8k {

constexpr uint32_t kMQChunk = 24576;
// ring A streams from HBM (96 KB in flight per SM); ring B mostly hits L2
// (the amax pass read the same bytes just before) but feeds the cast warps,
// whose chunks go fastest: of the splits of nine stages, 4/5 measured best
// (6/3 1.5% slower, 3/6 2%, 2/7 8%)
constexpr int kMQStagesA = 4, kMQStagesB = 5;
// warps reducing ring A / casting ring B: with 4 / 24 the amax stream fell
// to 3.5-4.4 TB/s while casts ran beside it (its 4 warps got few issue
// slots); 12 / 16 measured 36.5 against 38.5 us for the Float8 linear's
// three tensors (8 / 20 and 20 / 8: 38.5-38.6 us)
constexpr int kMQWarpsA = 12, kMQWarpsB = 16;
constexpr int kMQThreadsA = 32 * kMQWarpsA, kMQThreadsB = 32 * kMQWarpsB;
constexpr int kMQThreads = 64 + kMQThreadsA + kMQThreadsB;
constexpr int kMQNumBars = 2 * (kMQStagesA + kMQStagesB);
constexpr uint32_t kMQSmem = 1024 + (kMQStagesA + kMQStagesB) * kMQChunk + 8 * kMQNumBars + 64;

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void group_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Bounded wait until *ctr >= target (another CTA's release); false on timeout.
__device__ __forceinline__ bool wait_count(const uint32_t *ctr, uint32_t target,
                                           volatile int *abort, DevErr err, uint32_t where) {
  if (ld_acquire_gpu(ctr) >= target) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire_gpu(ctr) >= target) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > err.limit_ns) {
      *abort = 1;
      record_error(err, kErrTimeout, where);
      return false;
    }
  }
}

// The quantize warps' pass over one staged chunk of nvec 8-element vectors.
template <int F, typename T>
__device__ __forceinline__ void cast_chunk(const uint8_t *base, uint32_t nvec, uint2 *dst,
                                           const ScaleDiv &d, int tid) {
  if (d.fast) {
    // two vectors per step: independent FMA chains to interleave
    for (uint32_t v = tid; v < nvec; v += 2 * kMQThreadsB) {
      const uint32_t v2 = v + kMQThreadsB;
      Raw8<T> r0, r1;
      r0.load_shared(base + v * 8 * sizeof(T));
      if (v2 < nvec) r1.load_shared(base + v2 * 8 * sizeof(T));
      dst[v] = quant8_own_scale<F>(r0, d);
      if (v2 < nvec) dst[v2] = quant8_own_scale<F>(r1, d);
    }
  } else {
    for (uint32_t v = tid; v < nvec; v += kMQThreadsB) {
      Raw8<T> r;
      r.load_shared(base + v * 8 * sizeof(T));
      dst[v] = quant8_ieee<F>(r, d);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kMQThreads, 1)
    quant_multi_kernel(const __grid_constant__ MultiQuantArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *ring_a = smem;
  uint8_t *ring_b = smem + kMQStagesA * kMQChunk;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (kMQStagesA + kMQStagesB) * kMQChunk);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + kMQNumBars);
  __shared__ uint32_t red_a[kMQWarpsA];
  __shared__ float scale_b;

  auto full_a = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_a = [&](int s) { return smem_u32(&bars[kMQStagesA + s]); };
  auto full_b = [&](int s) { return smem_u32(&bars[2 * kMQStagesA + s]); };
  auto empty_b = [&](int s) { return smem_u32(&bars[2 * kMQStagesA + kMQStagesB + s]); };

  const uint32_t warp = threadIdx.x >> 5, lane = lane_id();
  const uint32_t G = gridDim.x, cta = blockIdx.x;
  const DevErr err{args.err, args.wait_limit_ns};
  uint32_t *keys = args.sync;
  uint32_t *done = args.sync + kMaxMulti;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMQStagesA; ++s) {
      mbar_init(full_a(s), 1);
      mbar_init(empty_a(s), kMQWarpsA);
    }
    for (int s = 0; s < kMQStagesB; ++s) {
      mbar_init(full_b(s), 1);
      mbar_init(empty_b(s), kMQWarpsB);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // chunk geometry of tensor t: bytes of whole 8-element vectors, chunk count
  auto vec_bytes = [&](int t) { return (uint64_t)(args.n[t] / 8) * 8 * sizeof(T); };
  auto chunks = [&](int t) { return (uint32_t)((vec_bytes(t) + kMQChunk - 1) / kMQChunk); };
  auto chunk_bytes = [&](int t, uint32_t c) {
    const uint64_t rest = vec_bytes(t) - (uint64_t)c * kMQChunk;
    return (uint32_t)(rest < kMQChunk ? rest : kMQChunk);
  };

  if (warp < 2) {
    // ------------------------------------------- producers (rings A and B)
    const bool is_a = (warp == 0);
    const int stages = is_a ? kMQStagesA : kMQStagesB;
    uint8_t *ring = is_a ? ring_a : ring_b;
    uint32_t it = 0;
    bool ok = true;
    for (int t = 0; t < args.count && ok; ++t) {
      const uint8_t *src = static_cast<const uint8_t *>(args.x[t]);
      for (uint32_t c = cta; c < chunks(t); c += G, ++it) {
        const int s = (int)(it % stages);
        const uint32_t round = it / stages;
        const uint32_t eb = is_a ? empty_a(s) : empty_b(s);
        const uint32_t fb = is_a ? full_a(s) : full_b(s);
        if (!mbar_wait_warp(eb, (round & 1u) ^ 1u, abort_flag, err, is_a ? 11 : 12)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t bytes = chunk_bytes(t, c);
          mbar_arrive_expect_tx(fb, bytes);
          bulk_load(smem_u32(ring + s * kMQChunk), src + (uint64_t)c * kMQChunk, bytes, fb);
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      // let the copies already issued land before the CTA can exit
      const uint32_t first = it > (uint32_t)stages ? it - stages : 0u;
      for (uint32_t i = first; i < it; ++i)
        drain_wait(is_a ? full_a(i % stages) : full_b(i % stages), (i / stages) & 1u);
    }
  } else if (warp < 2 + kMQWarpsA) {
    // ---------------------------------------------------- amax consumers
    const int tid = threadIdx.x - 64;
    uint32_t it = 0;
    for (int t = 0; t < args.count; ++t) {
      uint32_t key_a = 0, key_b = 0;
      for (uint32_t c = cta; c < chunks(t); c += G, ++it) {
        const int s = (int)(it % kMQStagesA);
        if (!mbar_wait_warp(full_a(s), (it / kMQStagesA) & 1u, abort_flag, err, 13)) continue;
        const uint32_t nvec = chunk_bytes(t, c) / (8 * sizeof(T));
        const uint8_t *base = ring_a + s * kMQChunk;
        // four vectors per step: four shared loads in flight per thread
        uint32_t v = tid;
        for (; v + 3 * kMQThreadsA < nvec; v += 4 * kMQThreadsA) {
          Raw8<T> r[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) r[u].load_shared(base + (v + u * kMQThreadsA) * 8 * sizeof(T));
#pragma unroll
          for (int u = 0; u < 4; ++u) r[u].max_abs(key_a, key_b);
        }
        for (; v < nvec; v += kMQThreadsA) {
          Raw8<T> r;
          r.load_shared(base + v * 8 * sizeof(T));
          r.max_abs(key_a, key_b);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_a(s));
      }
      uint32_t key = warp_max_u32(Raw8<T>::merge_keys(key_a, key_b));
      if (lane == 0) red_a[warp - 2] = key;
      group_sync(1, kMQThreadsA);
      if (tid == 0) {
        uint32_t k = 0;
        for (int w = 0; w < kMQWarpsA; ++w) k = max(k, red_a[w]);
        if (cta == 0) {  // elements after the last whole vector
          const T *x = static_cast<const T *>(args.x[t]);
          for (int64_t i = args.n[t] / 8 * 8; i < args.n[t]; ++i) k = max(k, abs_key(load1(x + i)));
        }
        atomicMax(keys + t, k);
        __threadfence();
        atomicAdd(done + t, 1u);
      }
      group_sync(1, kMQThreadsA);  // red_a is rewritten for the next tensor
    }
  } else {
    // ------------------------------------------------ quantize consumers
    const int tid = threadIdx.x - 64 - kMQThreadsA;
    uint32_t it = 0;
    for (int t = 0; t < args.count; ++t) {
      const int fmt = args.fmt[t];
      const float mx = fmt_max(fmt);
      if (tid == 0) {
        float s = 1.0f;
        if (wait_count(done + t, G, abort_flag, err, 14)) {
          const float amax = __uint_as_float(ld_acquire_gpu(keys + t));
          s = scale_from_amax(amax, mx);
          if (cta == 0) {
            if (args.amax_out[t] != nullptr) *args.amax_out[t] = amax;
            *args.scale_out[t] = s;
          }
        }
        scale_b = s;
      }
      group_sync(2, kMQThreadsB);
      const ScaleDiv d(scale_b);
      uint8_t *q = args.q[t];
      for (uint32_t c = cta; c < chunks(t); c += G, ++it) {
        const int s = (int)(it % kMQStagesB);
        if (!mbar_wait_warp(full_b(s), (it / kMQStagesB) & 1u, abort_flag, err, 15)) continue;
        const uint32_t nvec = chunk_bytes(t, c) / (8 * sizeof(T));
        const uint8_t *base = ring_b + s * kMQChunk;
        uint2 *dst = reinterpret_cast<uint2 *>(q + (uint64_t)c * (kMQChunk / sizeof(T)));
        if (fmt == 0)
          cast_chunk<0, T>(base, nvec, dst, d, tid);
        else
          cast_chunk<1, T>(base, nvec, dst, d, tid);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_b(s));
      }
      if (cta == 0 && tid == 0) {  // elements after the last whole vector
        const T *x = static_cast<const T *>(args.x[t]);
        for (int64_t i = args.n[t] / 8 * 8; i < args.n[t]; ++i) {
          const float y = d.div<false>(load1(x + i));
          q[i] = (uint8_t)(cvt_fp8x2(fmt, y, 0.0f) & 0xFFu);
        }
      }
      group_sync(2, kMQThreadsB);  // scale_b is rewritten for the next tensor
    }
  }
  __syncthreads();
}

cudaError_t launch_quant_multi(const MultiQuantArgs &args, int in_dt, int sms, cudaStream_t st) {
  auto kern_bf = quant_multi_kernel<__nv_bfloat16>;
  auto kern_f = quant_multi_kernel<float>;
  void *fn = in_dt == 0 ? reinterpret_cast<void *>(kern_bf) : reinterpret_cast<void *>(kern_f);
  static bool attr_done[64][2] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev][in_dt]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMQSmem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kMQThreads, kMQSmem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorLaunchOutOfResources;
    attr_done[dev][in_dt] = true;
  }
  e = cudaMemsetAsync(args.sync, 0, sizeof(uint32_t) * 2 * kMaxMulti, st);
  if (e != cudaSuccess) return e;
  // one CTA per SM, all co-resident (the quantize warps wait for every CTA)
  MultiQuantArgs a = args;
  void *params[] = {&a};
  return cudaLaunchCooperativeKernel(fn, dim3((unsigned)sms), dim3(kMQThreads), params, kMQSmem,
                                     st);
}

}  // namespace fp8k
