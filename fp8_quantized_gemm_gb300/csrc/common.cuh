// Shared device helpers for the sm_103a kernels: inline-PTX wrappers for
// mbarriers, TMA (cp.async.bulk.tensor), tcgen05 (TMEM alloc, MMA, commit,
// ld/st, cp) and FP8 conversion, plus the bounded-wait policy.
//
// Every spin on an mbarrier is bounded by %globaltimer: after the wait limit
// (kWaitLimitNs by default; settable per call through the error-word struct,
// which the failure tests use to make waits run out) the waiter records FP8_ERR_TIMEOUT in the library's device error word, raises a
// CTA-wide abort flag in shared memory (so the other roles stop waiting too)
// and returns false; the kernel then runs its normal teardown (TMEM dealloc)
// and exits.  Nothing here traps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8k {

constexpr float kE4M3Max = 448.0f;
constexpr float kE5M2Max = 57344.0f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr uint32_t kErrTimeout = 5;               // stored as -FP8_ERR_TIMEOUT

__device__ __forceinline__ float fmt_max(int fmt) { return fmt == 0 ? kE4M3Max : kE5M2Max; }

// ------------------------------------------------------------ error word --
struct DevErr {
  uint32_t *word;     // [0] = first error code (positive), [1] = where
  uint64_t limit_ns;  // bound of every wait
};

__device__ __forceinline__ void record_error(DevErr e, uint32_t code, uint32_t where) {
  if (e.word != nullptr && atomicCAS(e.word, 0u, code) == 0u) e.word[1] = where;
}

// ----------------------------------------------------------------- misc --
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// -------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrival without release semantics (see mbar_arrive_cluster_relaxed).
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `bar` with parity `parity` to complete.
// Returns false (after recording the timeout and raising *abort) when the
// limit expires, or when another role has already raised *abort.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          DevErr err, uint32_t where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > err.limit_ns) {
      *abort = 1;
      record_error(err, kErrTimeout, where);
      return false;
    }
  }
}

// mbar_wait for a whole warp: every lane calls it; the result is the same on
// all lanes (a lane that gave up makes the warp give up), so warp-collective
// instructions after it (elect.sync, tcgen05.ld .sync.aligned) never run on a
// partial warp.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int *abort,
                                               DevErr err, uint32_t where) {
  const bool ok = mbar_wait(bar, parity, abort, err, where);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Short non-abortable wait used only on the abort path (drains async work
// before the CTA exits).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 20000000ull) break;  // 20 ms
  }
}

// A fixed pause (abort paths only): lets copies that no barrier of this CTA
// tracks land before it exits.
__device__ __forceinline__ void grace_wait(uint64_t ns) {
  const uint64_t t0 = globaltimer();
  while (globaltimer() - t0 < ns) __nanosleep(1000);
}

// -------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Bring one tensor-map box into L2 (no shared-memory destination, no
// completion to wait for): a hint that warms the cache for a later load.
// Bring the line holding p into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *m, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1)
               : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before the previous kernel in the stream has
// finished.  grid_dependency_wait() blocks the calling thread until that
// kernel has completed and its memory operations are visible (a no-op when
// there is none); launch_dependents() lets the next such kernel start once
// every CTA of this one has called it or exited.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// TMA load delivered to the same shared-memory offset in every CTA of the
// cluster named by `mask`; each destination's mbarrier at `bar`'s offset
// receives the bytes it got.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                               int32_t c0, int32_t c1, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar), "h"(mask)
      : "memory");
}

// TMA store of one tensor-map box from shared memory (bulk-group
// completion: commit, then wait on the group).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, uint32_t src, int32_t c0,
                                             int32_t c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
// The same with an L2 eviction-priority hint (a createpolicy value):
// results that nothing in the kernel reads again are stored evict-first so
// they do not push the operands out of L2.
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap *m, uint32_t src, int32_t c0,
                                                  int32_t c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint"
      " [%0, {%1, %2}], [%3], %4;" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(c0), "r"(c1), "r"(src), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups still read their shared source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk group has completed (writes done).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------------- tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row atoms of 1024 bytes.
// Fields: start address >> 4 (bits 0-13), leading byte offset >> 4 (16-29,
// unused for swizzled K-major, set to 1), stride byte offset >> 4 (32-45:
// 1024 bytes between 8-row atoms), descriptor version 1 (bits 46-47),
// base offset 0 (tile base 1024-aligned), layout SWIZZLE_128B = 2 (61-63).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr) {
  return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Shared-memory matrix descriptor for an MN-major operand tile written by
// TMA with 128-byte swizzling (box {128 rows of the operand, 128 K}): each
// 128-byte line holds 128 consecutive M (or N) elements of one K index, 8
// lines form a 1024-byte atom, atoms follow each other along K (stride byte
// offset 1024), and further 128-element blocks of M or N sit `lbo` bytes
// apart (leading byte offset).  One K = 32 step of the MMA covers four atoms,
// so the start address advances by 4096 bytes per step.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t smem_addr, uint32_t lbo) {
  return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Operand descriptor and its per-K=32-step increment (in 16-byte units) for
// either layout: K-major steps 32 bytes along the swizzled line, MN-major
// steps four 1024-byte atoms.
struct OperandDesc {
  uint64_t base;
  uint32_t step;
};
__device__ __forceinline__ OperandDesc operand_desc(uint32_t smem_addr, int mn_major,
                                                    uint32_t mn_lbo) {
  if (mn_major) return {sdesc_sw128_mn(smem_addr, mn_lbo), 4096u >> 4};
  return {sdesc_sw128(smem_addr), 32u >> 4};
}

// Descriptor of an unswizzled K-major source for tcgen05.cp: 8-row x 16-byte
// core matrices stored contiguously (row stride 16 bytes, 128 bytes apart).
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t smem_addr) {
  return (uint64_t)((smem_addr >> 4) & 0x3FFFu) | ((uint64_t)(128 >> 4) << 16) |
         ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor, kind::f8f6f4 (dense): D = f32 (bits 4-5 = 1),
// A/B formats at bits 7-9 / 10-12 (E4M3 = 0, E5M2 = 1), A / B major-ness at
// bits 15 / 16 (0 = K-major, 1 = MN-major), N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f8f6f4(uint32_t m, uint32_t n, uint32_t fa,
                                                    uint32_t fb, uint32_t a_mn = 0,
                                                    uint32_t b_mn = 0) {
  return (1u << 4) | (fa << 7) | (fb << 10) | (a_mn << 15) | (b_mn << 16) | ((n >> 3) << 17) |
         ((m >> 4) << 24);
}

// Instruction descriptor, kind::mxf8f6f4 with block scaling: B scale-factor
// id at bits 4-5, formats at 7-9 / 10-12, N >> 3 at 17-22, scale type UE8M0
// (bit 23 = 1), M >> 4 at 24-28, A scale-factor id at bits 29-30.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4(uint32_t m, uint32_t n, uint32_t fa,
                                                      uint32_t fb, uint32_t sfa_id,
                                                      uint32_t sfb_id) {
  return (sfb_id << 4) | (fa << 7) | (fb << 10) | ((n >> 3) << 17) | (1u << 23) |
         ((m >> 4) << 24) | (sfa_id << 29);
}

__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t sfa_tmem,
                                             uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` when every tcgen05 op this thread issued so far completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// mma_commit that arrives on the mbarrier at the same offset in every CTA of
// the cluster named by `mask` (a cluster whose CTAs share operand tiles).
__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// smem (32 rows x 16 bytes) -> TMEM 32 lanes x 4 columns, replicated into all
// four 32-lane sub-partitions.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

#define FP8K_TMEM_LD_X32(taddr, r)                                                            \
  asm volatile(                                                                               \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"       \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),   \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),            \
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),         \
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),         \
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),         \
        "=r"(r[31])                                                                           \
      : "r"(taddr))

#define FP8K_TMEM_LD_X16(taddr, r)                                                            \
  asm volatile(                                                                               \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
      "%14,%15}, [%16];"                                                                      \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),   \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),            \
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])                                                 \
      : "r"(taddr))

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// An empty volatile statement that "rewrites" 16 registers: placed after
// tcgen05.wait::ld, it keeps every use of those tcgen05.ld results after the
// wait in the compiler's order (no instruction is emitted).
#define FP8K_REG_FENCE16(r)                                                                  \
  asm volatile(""                                                                            \
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),     \
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),   \
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]))

// ------------------------------------------- CTA pairs (cta_group::2) --
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cta address -> shared::cluster address of the same offset in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store four consecutive floats to another CTA's shared memory (16-byte
// aligned shared::cluster address); made visible to that CTA by a cluster
// barrier's release / acquire.
__device__ __forceinline__ void st_shared_cluster_v4(uint32_t cluster_addr, float a, float b,
                                                     float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "f"(a),
               "f"(b), "f"(c), "f"(d)
               : "memory");
}

// arrive on an mbarrier anywhere in the cluster (shared::cluster address)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// The same arrival without release semantics: it orders none of the
// thread's earlier memory operations (a release at cluster scope waits for
// every load and store still in flight).  For hand-backs whose only
// precondition is already complete, e.g. TMEM reads after tcgen05.wait::ld.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// TMA load into this CTA's shared memory, completing on an mbarrier that may
// sit in the peer CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *m,
                                                 uint32_t bar_cluster, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}

// M = 256 MMA over the CTA pair: A rows split 128/128 and B rows (N) split
// half/half between the two CTAs' shared memory at the same offsets; each
// CTA's TMEM receives its 128 rows of D.
__device__ __forceinline__ void mma_f8f6f4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at the same offset in every CTA of `mask` when the
// pair's tcgen05 ops issued so far complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// ------------------------------------------------------------ conversion --
// Two fp32 -> two FP8 codes, round to nearest even, saturating to +-MAX.
// PTX places the first source operand in the UPPER byte, so `hi` is the
// element at the higher address.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t cvt_e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t cvt_fp8x2(int fmt, float lo, float hi) {
  return fmt == 0 ? cvt_e4m3x2(lo, hi) : cvt_e5m2x2(lo, hi);
}

// Quantize one value: fl32(x / s); the clip to +-MAX is done by the
// saturating conversion (cvt.rn.satfinite rounds to nearest even and clamps
// finite values beyond the largest finite code to it, which for every finite
// y equals rounding clip(y, -MAX, MAX)).
//
// Many values are divided by one scale, so the quotient is formed from the
// correctly rounded reciprocal y = RN(1/s) by Markstein's FMA correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990; J.-M. Muller et al.,
// Handbook of Floating-Point Arithmetic, division with an FMA):
//   q0 = RN(x y)             within 2 ulp of z = x / s (|y s - 1| < 2^-24);
//   q1 = RN(q0 + RN(x - s q0) y)   within 2^-22 ulp of z before rounding,
//                                  hence a faithful rounding of z;
//   q2 = RN(q1 + (x - s q1) y)     the remainder x - s q1 is exact because q1
//                                  is faithful, and a quotient of two binary32
//                                  numbers lies more than 2^-25 ulp from any
//                                  midpoint, farther than the correction errs,
//                                  so q2 = RN(z).
// Preconditions, checked once per scale (ScaleDiv::fast): s in [2^-80, 2^80],
// which keeps y normal and every remainder that matters (|z| >= 2^-23) free
// of underflow.  Quotients below 2^-23 may differ from RN(z) in their last
// bits but round to a signed zero in both FP8 formats either way, and the
// sign is copied from x, as IEEE division gives it.  For |q0| >= 2^100 (x
// infinite, or a quotient far beyond either format's MAX) and NaN x, q0 is
// kept: the conversion saturates it, or keeps the NaN, as it would RN(z).
__device__ __forceinline__ float div_by_scale(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r0 = __fmaf_rn(-s, q0, x);
  const float q1 = __fmaf_rn(r0, y, q0);
  const float r1 = __fmaf_rn(-s, q1, x);
  const float q2 = copysignf(__fmaf_rn(r1, y, q1), x);
  return fabsf(q0) < 0x1p100f ? q2 : q0;
}

// Packed fp32 pairs for the f32x2 FMA pipe of sm_100-class GPUs (one
// instruction computes two independent single-precision mul / fma, each
// rounded as the scalar instruction would be).
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// div_by_scale on two values at once: the same five rounded operations per
// value, issued as packed pairs (y2 = {y, y}, ns2 = {-s, -s}).
__device__ __forceinline__ void div_by_scale2(float x0, float x1, uint64_t ns2, uint64_t y2,
                                              float &o0, float &o1) {
  const uint64_t xv = f32x2_pack(x0, x1);
  const uint64_t q0 = f32x2_mul(xv, y2);
  const uint64_t r0 = f32x2_fma(ns2, q0, xv);
  const uint64_t q1 = f32x2_fma(r0, y2, q0);
  const uint64_t r1 = f32x2_fma(ns2, q1, xv);
  const uint64_t q2 = f32x2_fma(r1, y2, q1);
  float a0, a1, b0, b1;
  f32x2_unpack(q0, a0, a1);
  f32x2_unpack(q2, b0, b1);
  o0 = fabsf(a0) < 0x1p100f ? copysignf(b0, x0) : a0;
  o1 = fabsf(a1) < 0x1p100f ? copysignf(b1, x1) : a1;
}

// div_by_scale2 for quotients known to be finite and far from overflow (the
// scale was formed from this very tensor's amax, so |x / s| <= MAX (1 +
// 2^-23) and x is finite): no range guard, and the sign is not forced.  A
// positive x still gives a non-negative result and a negative x a
// non-positive one, but a zero or underflowed quotient may carry the wrong
// sign of zero; the caller puts x's sign into each FP8 code instead.
__device__ __forceinline__ void div_by_scale2_bounded(float x0, float x1, uint64_t ns2,
                                                      uint64_t y2, float &o0, float &o1) {
  const uint64_t xv = f32x2_pack(x0, x1);
  const uint64_t q0 = f32x2_mul(xv, y2);
  const uint64_t r0 = f32x2_fma(ns2, q0, xv);
  const uint64_t q1 = f32x2_fma(r0, y2, q0);
  const uint64_t r1 = f32x2_fma(ns2, q1, xv);
  f32x2_unpack(f32x2_fma(r1, y2, q1), o0, o1);
}

struct ScaleDiv {
  float s, y;
  uint64_t ns2, y2;  // {-s, -s}, {y, y} for div_by_scale2
  // fast path: a magnitude from which on x / s saturates every FP8 format
  // and up to which the quotient stays below 2^64 (no overflow): s 2^64,
  // or 2^127 once that is larger (s > 2^63; with s <= 2^80, 2^127 / s >=
  // 2^47, far beyond either format's MAX)
  float bound;
  bool fast;
  __device__ __forceinline__ explicit ScaleDiv(float s_) {
    s = s_;
    y = __frcp_rn(s_);
    ns2 = f32x2_pack(-s_, -s_);
    y2 = f32x2_pack(y, y);
    bound = fminf(__fmul_rn(s_, 0x1p64f), 0x1p127f);
    fast = s_ >= 0x1p-80f && s_ <= 0x1p80f;
  }
  // kFast: the caller has checked `fast` (uniformly, outside its loop)
  template <bool kFast>
  __device__ __forceinline__ float div(float x) const {
    if constexpr (kFast)
      return div_by_scale(x, s, y);
    else
      return __fdiv_rn(x, s);
  }
  // eight quotients (four packed pairs on the fast path)
  template <bool kFast>
  __device__ __forceinline__ void div8(const float (&v)[8], float (&o)[8]) const {
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      if constexpr (kFast) {
        div_by_scale2(v[j], v[j + 1], ns2, y2, o[j], o[j + 1]);
      } else {
        o[j] = __fdiv_rn(v[j], s);
        o[j + 1] = __fdiv_rn(v[j + 1], s);
      }
    }
  }
};

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// |x| as an order-preserving uint32 key (non-negative floats order like uints).
__device__ __forceinline__ uint32_t abs_key(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// fp32 scale from an amax: fl32(amax / MAX), or 1.0 for amax == 0.
__device__ __forceinline__ float scale_from_amax(float amax, float mx) {
  return amax > 0.0f ? __fdiv_rn(amax, mx) : 1.0f;
}

// Exact ceil(log2(s)) for finite s > 0 (normal or subnormal fp32).
__device__ __forceinline__ int ceil_log2_pos(float s) {
  const uint32_t b = __float_as_uint(s);
  const int ef = (int)(b >> 23);
  const uint32_t man = b & 0x7FFFFFu;
  if (ef != 0) return (ef - 127) + (man != 0u ? 1 : 0);
  // subnormal: s = man * 2^-149; ceil(log2) = floor(log2(man)) - 149 (+1 unless pow2)
  const int fl = 31 - __clz((int)man);
  return fl - 149 + ((man & (man - 1u)) != 0u ? 1 : 0);
}

// 2^e as fp32 for e in [-149, 127].
__device__ __forceinline__ float exp2_int(int e) {
  if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
  return __uint_as_float(1u << (e + 149));
}

}  // namespace fp8k
