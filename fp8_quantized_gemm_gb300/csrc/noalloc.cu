// fp8_gemm_group_noalloc: the per-K-group GEMM for callers that cannot
// allocate device memory.
//
// The regular fp8_gemm_group allocates device memory on first use for some
// shapes (the E8M0-word buffer of UE8M0 scales beyond one row tile).  Some
// callers cannot allow that: runtimes that reserve all device memory up
// front in their own pool, and code that must never stall on the allocator
// (cudaMalloc and cudaFree may synchronize the device).  This entry point
// always runs the tensor-core per-group kernel; where that kernel splits K
// for small M it keeps the fp32 partial sums and per-tile arrival counters in
// a fixed scratch array compiled into the library -- 64 KiB of counters plus
// 8 MiB of partials, held on every GPU that loads the library until the
// process exits -- and reduces them in global memory (the workspace form of
// the split).  It allocates nothing.
#include <nvtx3/nvToolsExt.h>

#include <mutex>

#include "fp8gemm.h"
#include "kernels.h"

namespace fp8k {
int api_device(int *sms, uint32_t **err);
int api_encode_operand(CUtensorMap *map, const void *base, int64_t k, int64_t rows, int box_rows);
}  // namespace fp8k

namespace {

constexpr size_t kCounterBytes = 64 * 1024;      // uint32 arrival counter per output tile
constexpr size_t kPartialBytes = 8u << 20;       // fp32 partials [ksplit][M][N]
constexpr size_t kScratchBytes = kCounterBytes + kPartialBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
unsigned char *g_scratch_ptr[64] = {};

// Device address of the scratch array for the current device.  In host code
// `g_noalloc_scratch` names a host-side stand-in, not device memory, so the
// address is looked up once per device with that device current.
int scratch_for_current_device(unsigned char **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return FP8_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<unsigned char *>(p);
  }
  *out = g_scratch_ptr[dev];
  return FP8_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace {

int gemm_group_noalloc(const uint8_t *a, const void *sa, const uint8_t *b, const void *sb,
                       int sfmt, int64_t M, int64_t N, int64_t K, void *c, int64_t ldc,
                       fp8_stream_t stream) {
  if (a == nullptr || b == nullptr || sa == nullptr || sb == nullptr || c == nullptr)
    return FP8_ERR_INVALID_ARG;
  if (sfmt != FP8_SCALE_F32 && sfmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
  const int64_t kMaxDim = (int64_t)1 << 31;
  if (M < 1 || N < 1 || K < 1 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim || ldc < N)
    return FP8_ERR_INVALID_ARG;
  if (K % 128 != 0 || !aligned16(a) || !aligned16(b) || (reinterpret_cast<uintptr_t>(c) & 1u))
    return FP8_ERR_MISALIGNED;

  int sms = 0;
  uint32_t *err = nullptr;
  int rc = fp8k::api_device(&sms, &err);
  if (rc != FP8_OK) return rc;
  unsigned char *scratch = nullptr;
  if ((rc = scratch_for_current_device(&scratch)) != FP8_OK) return rc;

  const int mode = sfmt == FP8_SCALE_F32 ? fp8k::kScaleGroupF32 : fp8k::kScaleGroupUe8m0;
  const int bn = fp8k::gemm_tile_n(mode, M, N, sms);
  fp8k::GemmArgs args{};
  args.M = M; args.N = N; args.K = K; args.fa = FP8_E4M3; args.fb = FP8_E4M3;
  args.out_dt = FP8_OUT_BF16; args.ldc = ldc; args.c = c; args.sa = sa; args.sb = sb;
  args.err = err;
  args.wait_limit_ns = fp8k::wait_limit_ns();
  args.vec_store = (aligned16(c) && (ldc * 2) % 16 == 0) ? 1 : 0;
  // split K through the fixed scratch (partials in global memory), not a
  // cluster: this entry point keeps the workspace form of the reduction
  args.ksplit = fp8k::gemm_ksplit(mode, M, N, K, sms, false);
  args.cluster_split = 0;
  const cudaStream_t st = (cudaStream_t)stream;
  if (args.ksplit > 1) {
    const int64_t tiles = ((M + 127) / 128) * ((N + bn - 1) / bn);
    const size_t partials = (size_t)args.ksplit * (size_t)M * (size_t)N * sizeof(float);
    if (partials > kPartialBytes || (size_t)tiles * 4 > kCounterBytes) return FP8_ERR_SCRATCH_LIMIT;
    args.counters = reinterpret_cast<uint32_t *>(scratch);
    args.ws = reinterpret_cast<float *>(scratch + kCounterBytes);
    // the array keeps the previous call's contents: counters must start at 0
    if (cudaMemsetAsync(args.counters, 0, (size_t)tiles * 4, st) != cudaSuccess)
      return FP8_ERR_CUDA;
  }
  CUtensorMap tma, tmb;
  if ((rc = fp8k::api_encode_operand(&tma, a, K, M, 128)) != FP8_OK) return rc;
  if ((rc = fp8k::api_encode_operand(&tmb, b, K, N, bn)) != FP8_OK) return rc;
  return fp8k::launch_gemm(mode, tma, tmb, args, sms, st) == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace

extern "C" int fp8_gemm_group_noalloc(const uint8_t *a, const void *sa, const uint8_t *b,
                                      const void *sb, int sfmt, int64_t M, int64_t N, int64_t K,
                                      void *c, int64_t ldc, fp8_stream_t stream) {
  nvtxRangePushA("fp8_gemm_group_noalloc");
  const int rc = gemm_group_noalloc(a, sa, b, sb, sfmt, M, N, K, c, ldc, stream);
  nvtxRangePop();
  return rc;
}
