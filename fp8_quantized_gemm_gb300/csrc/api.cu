// C ABI of libfp8gemm.so (declared in include/fp8gemm.h): argument
// validation, TMA descriptor encoding, per-device setup and launches.
//
// The library links the CUDA runtime statically and reaches the driver's
// cuTensorMapEncodeTiled through cudaGetDriverEntryPointByVersion, so the
// shared object loads on a machine without a GPU driver (only the calls need
// a device).
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <map>
#include <tuple>
#include <mutex>
#include <utility>

#include "fp8gemm.h"
#include "kernels.h"
#include "support.h"

namespace {

using fp8k::GemmArgs;

// An NVTX range named after the entry point around each call, so that a
// timeline shows which library call enqueued which kernels (NVTX v3 is
// header-only: without a profiler attached the range is a no-op).
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

// Device error word: [0] first error code (positive), [1] where.
__device__ uint32_t g_device_error[2];

struct DeviceState {
  bool ready = false;
  int sms = 0;
  uint32_t *err = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

// Device workspace of the UE8M0 per-group GEMM beyond one row tile: the
// E8M0 words the byte scales are expanded into (see fp8_gemm_group_bias),
// one buffer per (device, stream, slot) so that calls on different streams
// never share it.  Allocated on first need and grown by doubling; never
// inside a stream capture.  (Split K needs no workspace: the splits of a
// tile reduce inside a thread-block cluster.)
struct Workspace {
  void *ptr = nullptr;
  size_t bytes = 0;
};
constexpr int kWsWords = 1;
std::map<std::tuple<int, cudaStream_t, int>, Workspace> g_ws;

// CTA-pair GEMM path switch (on by default; fp8_set_option turns it off).
bool g_use_pairs = true;
// B-multicast clusters in the single-CTA GEMM (on by default).
bool g_use_multicast = true;
// TMA-store epilogue of the CTA-pair GEMM (off by default: once the
// accumulator hand-back stopped waiting on the warp's stores, plain stores
// measured 69.1 us on the Float8 linear's grouped launch against 70.2-73.3 us
// through the TMA-store epilogue).
bool g_use_tma_store = false;
// CUDA-core path of the per-group GEMM for one row (off by default: inside
// CUDA graphs the few-row tensor-core kernel measured faster, 5.7 against
// 6.5 us at N 2048, K 7168, as it overlaps its start with the previous
// kernel; single launches are about equal).
bool g_use_gemv = false;
// Few-row tensor-core kernel of the per-group GEMM (on by default).
bool g_use_skinny = true;
// 256-row tiles per band of the CTA-pair kernel's tile order.
int64_t g_pair_band_rows = 8;
// Bound of every device-side mbarrier wait (fp8_set_option).
uint64_t g_wait_limit_ns = 2000000000ull;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int to_status(cudaError_t e) { return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA; }

// Per-device setup, once per device with that device current.
int device_state(DeviceState **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FP8_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return FP8_ERR_NO_DEVICE;  // built for sm_103a only
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FP8_ERR_CUDA;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return FP8_ERR_CUDA;
    d.err = static_cast<uint32_t *>(p);
    if (g_encode == nullptr) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return FP8_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return FP8_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_fmt(int f) { return f == FP8_E4M3 || f == FP8_E5M2; }
bool valid_in(int d) { return d == FP8_IN_BF16 || d == FP8_IN_F32; }
constexpr int64_t kMaxDim = (int64_t)1 << 31;

// 2-D uint8 operand [rows, k] with row pitch k bytes; box {128, box_rows},
// 128-byte swizzle (the layout the UMMA shared-memory descriptor expects).
int encode_operand(CUtensorMap *map, const void *base, int64_t k, int64_t rows, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)k};
  const cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

// 2-D uint8 operand stored MN-major, [k, rows] with row pitch `rows` bytes:
// box {128 rows of the operand, 128 K}, 128-byte swizzle.
int encode_operand_mn(CUtensorMap *map, const void *base, int64_t k, int64_t rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)rows, (cuuint64_t)k};
  const cuuint64_t strides[1] = {(cuuint64_t)rows};
  const cuuint32_t box[2] = {128u, 128u};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

// Tensor map of a per-tensor GEMM operand in either layout (box_rows: the
// K-major box height the kernel stages).
int encode_gemm_operand(CUtensorMap *map, const void *base, int mn_major, int64_t k,
                        int64_t rows, int box_rows) {
  return mn_major ? encode_operand_mn(map, base, k, rows)
                  : encode_operand(map, base, k, rows, box_rows);
}

// Output C [M, N] (pitch ldc elements) for the CTA-pair kernel's TMA-store
// epilogue: boxes of 32 rows x 128 bytes (64 bf16 or 32 fp32), 128-byte
// swizzle.  Needs a 16-byte aligned base and pitch.
int encode_output(CUtensorMap *map, void *c, int out_dt, int64_t M, int64_t N, int64_t ldc) {
  const cuuint64_t es = out_dt == FP8_OUT_F32 ? 4 : 2;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)ldc * es};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / es), 32u};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = g_encode(map,
                        out_dt == FP8_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                              : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        2, c, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

int check_output(const void *c, int64_t N, int64_t ldc, int out_dt) {
  if (c == nullptr) return FP8_ERR_INVALID_ARG;
  if (out_dt != FP8_OUT_F32 && out_dt != FP8_OUT_BF16) return FP8_ERR_INVALID_ARG;
  if (ldc < N) return FP8_ERR_INVALID_ARG;
  const uintptr_t es = out_dt == FP8_OUT_F32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(c) & (es - 1)) != 0) return FP8_ERR_MISALIGNED;
  return FP8_OK;
}

// 16-byte vector stores need an aligned base and a row pitch of 16-byte multiples.
int vector_store_ok(const void *c, int64_t ldc, int out_dt) {
  const int64_t es = out_dt == FP8_OUT_F32 ? 4 : 2;
  return aligned16(c) && (ldc * es) % 16 == 0 ? 1 : 0;
}

// Whether the CTA-pair epilogue may write C with TMA stores (plain stores
// otherwise: accumulation, or an unaligned base or pitch).
bool use_tma_store(const void *c, int64_t ldc, int out_dt, int accumulate) {
  return g_use_tma_store && accumulate == 0 && vector_store_ok(c, ldc, out_dt);
}

int get_workspace(cudaStream_t st, size_t need, void **out, int slot) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP8_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace &w = g_ws[std::make_tuple(dev, st, slot)];
  if (w.bytes < need) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return FP8_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return FP8_ERR_UNSUPPORTED;  // warm up before capture
    if (w.ptr != nullptr) {
      if (cudaStreamSynchronize(st) != cudaSuccess || cudaFree(w.ptr) != cudaSuccess)
        return FP8_ERR_CUDA;
      w.ptr = nullptr;
      w.bytes = 0;
    }
    size_t bytes = need > 2 * w.bytes ? need : 2 * w.bytes;
    bytes = (bytes + (1u << 20) - 1) & ~(size_t)((1u << 20) - 1);
    if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) return FP8_ERR_CUDA;
    if (cudaMemset(w.ptr, 0, bytes) != cudaSuccess) return FP8_ERR_CUDA;
    w.bytes = bytes;
  }
  *out = w.ptr;
  return FP8_OK;
}

int run_gemm(int mode, const uint8_t *a, const uint8_t *b, GemmArgs &args, cudaStream_t st) {
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  args.err = d->err;
  args.wait_limit_ns = g_wait_limit_ns;
  args.ksplit = fp8k::gemm_ksplit(mode, args.M, args.N, args.K, d->sms, true);
  args.ws = nullptr;
  args.counters = nullptr;
  // split K reduces inside a thread-block cluster (no workspace)
  args.cluster_split = args.ksplit > 1 ? 1 : 0;
  args.vec_store = vector_store_ok(args.c, args.ldc, args.out_dt);
  CUtensorMap tma, tmb;
  if ((rc = encode_gemm_operand(&tma, a, args.a_mn, args.K, args.M, 128)) != FP8_OK) return rc;
  if (args.ksplit == 1 && g_use_pairs && fp8k::gemm_pair_eligible(mode, args.M, args.N, d->sms)) {
    if ((rc = encode_gemm_operand(&tmb, b, args.b_mn, args.K, args.N,
                                  fp8k::gemm_pair_b_rows())) != FP8_OK)
      return rc;
    CUtensorMap tmc{};
    args.tma_store = use_tma_store(args.c, args.ldc, args.out_dt, args.accumulate) ? 1 : 0;
    if (args.tma_store &&
        (rc = encode_output(&tmc, args.c, args.out_dt, args.M, args.N, args.ldc)) != FP8_OK)
      return rc;
    return to_status(fp8k::launch_gemm_pair(tma, tmb, tmc, args, d->sms, st));
  }
  if (mode == fp8k::kScaleGroupF32 && args.ksplit == 1 && g_use_pairs && args.experts == 0 &&
      !args.a_mn && !args.b_mn &&
      fp8k::gemm_pair_promote_eligible(args.M, args.N, args.K, d->sms)) {
    if ((rc = encode_operand(&tmb, b, args.K, args.N, fp8k::gemm_pair_promote_b_rows())) != FP8_OK)
      return rc;
    return to_status(fp8k::launch_gemm_pair_promote(tma, tmb, args, d->sms, st));
  }
  // multicast pairs of vertically adjacent tiles share each B box: measured
  // faster for 128-wide tiles (the FP32-promotion mode, and the block-scaled
  // modes at mid-size M), not for the 128 x 256 block-scaled tiles
  const int bn = fp8k::gemm_tile_n(mode, args.M, args.N, d->sms);
  args.multicast = g_use_multicast && mode != fp8k::kScaleTensor &&
                           mode != fp8k::kScaleGroupF32x32 && bn == 128 &&
                           args.ksplit == 1 && !args.b_mn && args.experts == 0 && args.M > 128
                       ? 1
                       : 0;
  if ((rc = encode_gemm_operand(&tmb, b, args.b_mn, args.K, args.N,
                                args.multicast ? bn / 2 : bn)) != FP8_OK)
    return rc;
  return to_status(fp8k::launch_gemm(mode, tma, tmb, args, d->sms, st));
}

int check_gemm_common(const uint8_t *a, const uint8_t *b, int64_t M, int64_t N, int64_t K,
                      int64_t kgran) {
  if (a == nullptr || b == nullptr) return FP8_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim)
    return FP8_ERR_INVALID_ARG;
  if (K % kgran != 0 || !aligned16(a) || !aligned16(b)) return FP8_ERR_MISALIGNED;
  return FP8_OK;
}

// Validation of one per-tensor problem (fp8_gemm_tensor / _grouped).
int check_tensor_problem(const fp8_gemm_problem_t &p) {
  if (p.a == nullptr || p.b == nullptr) return FP8_ERR_INVALID_ARG;
  if (p.M < 1 || p.N < 1 || p.K < 1 || p.M >= kMaxDim || p.N >= kMaxDim || p.K >= kMaxDim)
    return FP8_ERR_INVALID_ARG;
  const bool lay_ok = (p.a_layout == FP8_K_MAJOR || p.a_layout == FP8_MN_MAJOR) &&
                      (p.b_layout == FP8_K_MAJOR || p.b_layout == FP8_MN_MAJOR);
  if (!lay_ok) return FP8_ERR_INVALID_ARG;
  if (p.sa == nullptr || p.sb == nullptr || !valid_fmt(p.fa) || !valid_fmt(p.fb))
    return FP8_ERR_INVALID_ARG;
  // the row pitch of each operand (K, or M / N when MN-major) must be a
  // multiple of 16 bytes for its tensor map
  const bool a_mn = p.a_layout == FP8_MN_MAJOR, b_mn = p.b_layout == FP8_MN_MAJOR;
  if (!aligned16(p.a) || !aligned16(p.b)) return FP8_ERR_MISALIGNED;
  if ((!a_mn || !b_mn) && p.K % 16 != 0) return FP8_ERR_MISALIGNED;
  if ((a_mn && p.M % 16 != 0) || (b_mn && p.N % 16 != 0)) return FP8_ERR_MISALIGNED;
  if (p.adamw != nullptr && p.swiglu != nullptr) return FP8_ERR_INVALID_ARG;
  if (p.adamw != nullptr) {
    const fp8_adamw_epilogue_t &e = *p.adamw;
    if (e.p == nullptr || e.m == nullptr || e.v == nullptr || e.step == nullptr)
      return FP8_ERR_INVALID_ARG;
    if (p.out_dt != FP8_OUT_F32 || p.accumulate != 0 || p.bias != nullptr || p.ldc < p.N)
      return FP8_ERR_UNSUPPORTED;
    if (!aligned16(e.p) || !aligned16(e.m) || !aligned16(e.v) || p.ldc % 4 != 0 ||
        (reinterpret_cast<uintptr_t>(e.p_bf16) & 7u) != 0 ||
        (reinterpret_cast<uintptr_t>(e.step) & 7u) != 0)
      return FP8_ERR_MISALIGNED;
    return FP8_OK;
  }
  int rc = check_output(p.c, p.N, p.ldc, p.out_dt);
  if (rc != FP8_OK) return rc;
  if (p.accumulate != 0 && (p.accumulate != 1 || p.out_dt != FP8_OUT_F32))
    return FP8_ERR_UNSUPPORTED;
  if (p.swiglu != nullptr) {
    const fp8_swiglu_epilogue_t &e = *p.swiglu;
    if (e.b_up == nullptr || e.sb_up == nullptr || e.u == nullptr || e.q == nullptr ||
        e.scale == nullptr || e.amax == nullptr || !valid_fmt(e.fmt))
      return FP8_ERR_INVALID_ARG;
    if (e.amax == e.scale) return FP8_ERR_INVALID_ARG;
    if (p.out_dt != FP8_OUT_BF16 || p.accumulate != 0 || p.bias != nullptr)
      return FP8_ERR_UNSUPPORTED;
    if (!aligned16(e.b_up) || !aligned16(e.u) || !aligned16(e.q) || !aligned16(p.c) ||
        p.N % 32 != 0 || p.ldc % 16 != 0)
      return FP8_ERR_MISALIGNED;
  }
  return FP8_OK;
}

// One validated per-tensor problem through the regular launch path.
int run_tensor_problem(const fp8_gemm_problem_t &p, cudaStream_t st) {
  GemmArgs args{};
  args.M = p.M; args.N = p.N; args.K = p.K; args.fa = p.fa; args.fb = p.fb;
  args.out_dt = p.out_dt; args.accumulate = p.accumulate; args.ldc = p.ldc; args.c = p.c;
  args.sa = p.sa; args.sb = p.sb;
  args.a_mn = p.a_layout == FP8_MN_MAJOR;
  args.b_mn = p.b_layout == FP8_MN_MAJOR;
  args.bias = p.bias;
  return run_gemm(fp8k::kScaleTensor, p.a, p.b, args, st);
}

}  // namespace

namespace fp8k {
uint64_t wait_limit_ns() { return g_wait_limit_ns; }
int64_t gemm_pair_band_rows() { return g_pair_band_rows; }

// Internal hooks for entry points defined in other files (noalloc.cu): the
// per-device setup (SM count, device error word) and the operand tensor map.
int api_device(int *sms, uint32_t **err) {
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  *sms = d->sms;
  *err = d->err;
  return FP8_OK;
}

int api_encode_operand(CUtensorMap *map, const void *base, int64_t k, int64_t rows, int box_rows) {
  return encode_operand(map, base, k, rows, box_rows);
}
}  // namespace fp8k

extern "C" {

int fp8_amax(const void *x, int in_dt, int64_t n, float *amax_out, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (amax_out == nullptr || n < 0 || !valid_in(in_dt) || (n > 0 && x == nullptr))
    return FP8_ERR_INVALID_ARG;
  if (n > 0 && !aligned16(x)) return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_amax(x, in_dt, n, amax_out, d->sms, (cudaStream_t)stream));
}

int fp8_quantize_tensor(const void *x, int in_dt, int64_t rows, int64_t cols, int fmt,
                        const float *amax_in, const float *scale, float *scale_out, uint8_t *q,
                        uint8_t *q_t, float *amax_out, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (x == nullptr || q == nullptr || !valid_in(in_dt) || !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (amax_in == nullptr && scale == nullptr) return FP8_ERR_INVALID_ARG;
  if (amax_out != nullptr && (amax_out == amax_in || amax_out == scale)) return FP8_ERR_INVALID_ARG;
  if (rows < 1 || cols < 1 || rows >= kMaxDim || cols >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (cols % 8 != 0 || !aligned16(x) || !aligned16(q) || (q_t != nullptr && !aligned16(q_t)))
    return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_quant_tensor(x, in_dt, rows, cols, fmt, amax_in, scale,
                                             scale_out, q, q_t, amax_out, d->sms,
                                             (cudaStream_t)stream));
}

int fp8_quantize_tensors(const fp8_quant_item_t *items, int count, uint32_t *sync,
                         fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  static_assert(FP8_QUANT_SYNC_WORDS == 2 * fp8k::kMaxMulti, "sync scratch size");
  if (items == nullptr || count < 1 || count > fp8k::kMaxMulti) return FP8_ERR_INVALID_ARG;
  if (sync == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned16(sync)) return FP8_ERR_MISALIGNED;
  const int in_dt = items[0].in_dt;
  if (!valid_in(in_dt)) return FP8_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    const fp8_quant_item_t &it = items[i];
    if (it.scale_out == nullptr || !valid_fmt(it.fmt)) return FP8_ERR_INVALID_ARG;
    if (!valid_in(it.in_dt)) return FP8_ERR_INVALID_ARG;
    if (it.in_dt != in_dt) return FP8_ERR_UNSUPPORTED;
    if (it.amax_out == it.scale_out) return FP8_ERR_INVALID_ARG;
    if (it.n < 0 || it.n >= ((int64_t)1 << 40)) return FP8_ERR_INVALID_ARG;
    // an empty tensor is read and written nowhere: its pointers may be null
    if (it.n > 0 && (it.x == nullptr || it.q == nullptr)) return FP8_ERR_INVALID_ARG;
    if (it.n > 0 && (!aligned16(it.x) || !aligned16(it.q))) return FP8_ERR_MISALIGNED;
  }
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  const cudaStream_t st = (cudaStream_t)stream;
  // The launch pipelines the tensors in order: the amax pass of the first
  // runs alone and so does the cast of the last.  The smallest tensor goes
  // first (the others keep their order): its short amax pass starts the
  // pipeline sooner.  Every tensor's outputs are its own, so the order does
  // not change any result.
  int order[fp8k::kMaxMulti], smallest = 0;
  for (int i = 1; i < count; ++i)
    if (items[i].n < items[smallest].n) smallest = i;
  order[0] = smallest;
  for (int i = 0, k = 1; i < count; ++i)
    if (i != smallest) order[k++] = i;
  fp8k::MultiQuantArgs a{};
  for (int j = 0; j < count; ++j) {
    const fp8_quant_item_t &it = items[order[j]];
    a.x[j] = it.x;
    a.n[j] = it.n;
    a.fmt[j] = it.fmt;
    a.q[j] = it.q;
    a.amax_out[j] = it.amax_out;
    a.scale_out[j] = it.scale_out;
  }
  a.count = count;
  a.sync = sync;
  a.err = d->err;
  a.wait_limit_ns = g_wait_limit_ns;
  return to_status(fp8k::launch_quant_multi(a, in_dt, d->sms, st));
}

int fp8_quantize_token_group(const void *x, int in_dt, int64_t M, int64_t K, int fmt, int sfmt,
                             uint8_t *q, void *scales, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (x == nullptr || q == nullptr || scales == nullptr || !valid_in(in_dt) || !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (sfmt != FP8_SCALE_F32 && sfmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
  if (M < 1 || K < 1 || M >= kMaxDim || K >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (K % 16 != 0 || !aligned16(x) || !aligned16(q)) return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_quant_group(x, in_dt, M, K, fmt, sfmt, q, scales, d->sms,
                                            (cudaStream_t)stream));
}

int fp8_quantize_block(const void *w, int in_dt, int64_t N, int64_t K, int fmt, int sfmt,
                       uint8_t *q, void *scales, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (w == nullptr || q == nullptr || scales == nullptr || !valid_in(in_dt) || !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (sfmt != FP8_SCALE_F32 && sfmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || N >= kMaxDim || K >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if ((N + 127) / 128 > 65535) return FP8_ERR_UNSUPPORTED;
  if (K % 16 != 0 || !aligned16(w) || !aligned16(q)) return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(
      fp8k::launch_quant_block(w, in_dt, N, K, fmt, sfmt, q, scales, (cudaStream_t)stream));
}

int fp8_quantize_mx(const void *x, int in_dt, int64_t R, int64_t K, int fmt, const float *amax,
                    float *global_out, uint8_t *q, uint32_t *local, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (x == nullptr || amax == nullptr || q == nullptr || local == nullptr || !valid_in(in_dt) ||
      !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (R < 1 || K < 1 || R >= kMaxDim || K >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (K % 128 != 0 || !aligned16(x) || !aligned16(q) || !aligned16(local))
    return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_quant_mx(x, in_dt, R, K, fmt, amax, global_out, q, local, d->sms,
                                         (cudaStream_t)stream));
}

int fp8_amax_rows(const void *x, int in_dt, int64_t R, int64_t K, float *amax_out,
                  fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (x == nullptr || amax_out == nullptr || !valid_in(in_dt)) return FP8_ERR_INVALID_ARG;
  if (R < 1 || K < 1 || R >= kMaxDim || K >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (K % 8 != 0 || !aligned16(x)) return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_row_amax(x, in_dt, R, K, amax_out, d->sms, (cudaStream_t)stream));
}

int fp8_quantize_mx_rows(const void *x, int in_dt, int64_t R, int64_t K, int fmt,
                         const float *amax_rows, float *global_out, uint8_t *q, uint32_t *local,
                         fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (x == nullptr || amax_rows == nullptr || global_out == nullptr || q == nullptr ||
      local == nullptr || !valid_in(in_dt) || !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (R < 1 || K < 1 || R >= kMaxDim || K >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (K % 128 != 0 || !aligned16(x) || !aligned16(q) || !aligned16(local))
    return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_quant_mx(x, in_dt, R, K, fmt, amax_rows, global_out, q, local,
                                         d->sms, (cudaStream_t)stream, true));
}

int fp8_quantize_mx1(const void *x, int in_dt, int64_t R, int64_t K, int fmt, float *global_out,
                     uint8_t *q, uint32_t *local, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (x == nullptr || q == nullptr || local == nullptr || !valid_in(in_dt) || !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (R < 1 || K < 1 || R >= kMaxDim || K >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (K % 128 != 0 || !aligned16(x) || !aligned16(q) || !aligned16(local))
    return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  // a null tensor amax selects the one-level variant of the two-level kernel
  return to_status(fp8k::launch_quant_mx(x, in_dt, R, K, fmt, nullptr, global_out, q, local,
                                         d->sms, (cudaStream_t)stream));
}

int fp8_quantize_block32(const void *w, int in_dt, int64_t N, int64_t K, int fmt, uint8_t *q,
                         uint8_t *scales, uint32_t *local, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (w == nullptr || q == nullptr || local == nullptr || !valid_in(in_dt) || !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || N >= kMaxDim || K >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (K % 128 != 0 || !aligned16(w) || !aligned16(q) || !aligned16(local))
    return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_quant_block32(w, in_dt, N, K, fmt, q, scales, local, d->sms,
                                              (cudaStream_t)stream));
}

int fp8_quantize_token_group32(const void *x, int in_dt, int64_t M, int64_t K, int fmt,
                               int sfmt, uint8_t *q, void *scales, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (x == nullptr || q == nullptr || scales == nullptr || !valid_in(in_dt) || !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (sfmt != FP8_SCALE_F32 && sfmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
  if (M < 1 || K < 1 || M >= kMaxDim || K >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (K % 16 != 0 || !aligned16(x) || !aligned16(q)) return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_quant_group32(x, in_dt, M, K, fmt, sfmt, q, scales, d->sms,
                                              (cudaStream_t)stream));
}

int fp8_quantize_block32_f32(const void *w, int in_dt, int64_t N, int64_t K, int fmt, uint8_t *q,
                             float *scales, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (w == nullptr || q == nullptr || scales == nullptr || !valid_in(in_dt) || !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || N >= kMaxDim || K >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (K % 32 != 0 || !aligned16(w) || !aligned16(q)) return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_quant_block32_f32(w, in_dt, N, K, fmt, q, scales, d->sms,
                                                  (cudaStream_t)stream));
}

int fp8_gemm_group32(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb,
                     int64_t M, int64_t N, int64_t K, void *c, int64_t ldc, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  int rc = check_gemm_common(a, b, M, N, K, 128);
  if (rc != FP8_OK) return rc;
  if (sa == nullptr || sb == nullptr) return FP8_ERR_INVALID_ARG;
  if ((rc = check_output(c, N, ldc, FP8_OUT_BF16)) != FP8_OK) return rc;
  GemmArgs args{};
  args.M = M; args.N = N; args.K = K; args.fa = FP8_E4M3; args.fb = FP8_E4M3;
  args.out_dt = FP8_OUT_BF16; args.ldc = ldc; args.c = c; args.sa = sa; args.sb = sb;
  return run_gemm(fp8k::kScaleGroupF32x32, a, b, args, (cudaStream_t)stream);
}

int fp8_dequantize_block(const uint8_t *q, int fmt, const void *scales, int sfmt, int64_t N,
                         int64_t K, void *out, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (q == nullptr || scales == nullptr || out == nullptr || !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (sfmt != FP8_SCALE_F32 && sfmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || N >= kMaxDim || K >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (K % 16 != 0 || (reinterpret_cast<uintptr_t>(q) & 7u) != 0 || !aligned16(out))
    return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(
      fp8k::launch_dequant_block(q, N, K, fmt, sfmt, scales, out, d->sms, (cudaStream_t)stream));
}

int fp8_gemm_tensor(const uint8_t *a, int fa, const uint8_t *b, int fb, const float *sa,
                    const float *sb, int64_t M, int64_t N, int64_t K, int out_dt, void *c,
                    int64_t ldc, int accumulate, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  fp8_gemm_problem_t p{};
  p.a = a; p.b = b; p.sa = sa; p.sb = sb; p.M = M; p.N = N; p.K = K; p.fa = fa; p.fb = fb;
  p.out_dt = out_dt; p.accumulate = accumulate; p.c = c; p.ldc = ldc;
  p.a_layout = FP8_K_MAJOR; p.b_layout = FP8_K_MAJOR;
  int rc = check_tensor_problem(p);
  if (rc != FP8_OK) return rc;
  return run_tensor_problem(p, (cudaStream_t)stream);
}

int fp8_gemm_tensor_grouped(const fp8_gemm_problem_t *problems, int count, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (problems == nullptr || count < 1 || count > 64) return FP8_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    const int rc = check_tensor_problem(problems[i]);
    if (rc != FP8_OK) return rc;
  }
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  const cudaStream_t st = (cudaStream_t)stream;
  // one persistent CTA-pair launch when every problem takes that path
  bool together = g_use_pairs && count <= fp8k::kMaxGroup;
  bool epilogue = false;
  int64_t tiles = 0;
  for (int i = 0; i < count; ++i) {
    const fp8_gemm_problem_t &p = problems[i];
    epilogue = epilogue || p.adamw != nullptr || p.swiglu != nullptr;
    together = together &&
               fp8k::gemm_ksplit(fp8k::kScaleTensor, p.M, p.N, p.K, d->sms, true) == 1;
    tiles += ((p.M + 255) / 256) * ((p.N + 255) / 256);
  }
  together = together && tiles * 4 >= d->sms / 2;
  // the epilogue variants live in the pair kernel, which takes any shape
  // (ragged tiles are masked): a group with one always runs there
  if (epilogue) {
    if (count > fp8k::kMaxGroup) return FP8_ERR_UNSUPPORTED;
    together = true;
  }
  if (!together) {
    for (int i = 0; i < count; ++i)
      if ((rc = run_tensor_problem(problems[i], st)) != FP8_OK) return rc;
    return FP8_OK;
  }
  // longest K first: the strided tile assignment then balances the pairs
  int order[fp8k::kMaxGroup];
  for (int i = 0; i < count; ++i) order[i] = i;
  for (int i = 1; i < count; ++i)
    for (int j = i; j > 0 && problems[order[j]].K > problems[order[j - 1]].K; --j) {
      const int tmp = order[j];
      order[j] = order[j - 1];
      order[j - 1] = tmp;
    }
  CUtensorMap tma[fp8k::kMaxGroup], tmb[fp8k::kMaxGroup], tmc[fp8k::kMaxGroup] = {};
  CUtensorMap tmb2[fp8k::kMaxGroup] = {};
  bool any_gated = false;
  GemmArgs args[fp8k::kMaxGroup];
  for (int k = 0; k < count; ++k) {
    const fp8_gemm_problem_t &p = problems[order[k]];
    GemmArgs a{};
    a.M = p.M; a.N = p.N; a.K = p.K; a.fa = p.fa; a.fb = p.fb; a.out_dt = p.out_dt;
    a.accumulate = p.accumulate; a.ldc = p.ldc; a.c = p.c; a.sa = p.sa; a.sb = p.sb;
    a.err = d->err;
    a.wait_limit_ns = g_wait_limit_ns;
    a.vec_store = vector_store_ok(p.c, p.ldc, p.out_dt);
    a.a_mn = p.a_layout == FP8_MN_MAJOR;
    a.b_mn = p.b_layout == FP8_MN_MAJOR;
    a.bias = p.bias;
    a.ksplit = 1;
    a.tma_store = use_tma_store(p.c, p.ldc, p.out_dt, p.accumulate) ? 1 : 0;
    if (p.adamw != nullptr) {
      const fp8_adamw_epilogue_t &e = *p.adamw;
      a.tma_store = 0;
      a.vec_store = 1;  // 16-byte aligned parameters and pitch (validated)
      a.adam_p = e.p;
      a.adam_m = e.m;
      a.adam_v = e.v;
      a.adam_pb = e.p_bf16;
      a.adam_step = e.step;
      a.adam_hp = fp8k::adamw_hp(e.lr, e.beta1, e.beta2, e.eps, e.weight_decay);
      a.adam_b1d = e.beta1;
      a.adam_b2d = e.beta2;
    }
    if (p.swiglu != nullptr) {
      const fp8_swiglu_epilogue_t &e = *p.swiglu;
      a.tma_store = 0;
      a.gated = 1;
      a.swi_sb2 = e.sb_up;
      a.swi_u = e.u;
      a.swi_q = e.q;
      a.swi_scale = e.scale;
      a.swi_amax = reinterpret_cast<uint32_t *>(e.amax);
      a.swi_fmt = e.fmt;
      any_gated = true;
      if ((rc = encode_gemm_operand(&tmb2[k], e.b_up, a.b_mn, p.K, p.N,
                                    fp8k::gemm_pair_b_rows())) != FP8_OK)
        return rc;
    }
    if (a.tma_store && (rc = encode_output(&tmc[k], p.c, p.out_dt, p.M, p.N, p.ldc)) != FP8_OK)
      return rc;
    args[k] = a;
    if ((rc = encode_gemm_operand(&tma[k], p.a, a.a_mn, p.K, p.M, 128)) != FP8_OK) return rc;
    if ((rc = encode_gemm_operand(&tmb[k], p.b, a.b_mn, p.K, p.N, fp8k::gemm_pair_b_rows())) !=
        FP8_OK)
      return rc;
  }
  return to_status(fp8k::launch_gemm_pair_group(tma, tmb, tmc, any_gated ? tmb2 : nullptr, args,
                                                count, d->sms, st));
}

int fp8_gemm_group(const uint8_t *a, const void *sa, const uint8_t *b, const void *sb, int sfmt,
                   int64_t M, int64_t N, int64_t K, void *c, int64_t ldc, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  return fp8_gemm_group_bias(a, sa, b, sb, sfmt, M, N, K, nullptr, c, ldc, stream);
}

int fp8_gemm_group_bias(const uint8_t *a, const void *sa, const uint8_t *b, const void *sb,
                        int sfmt, int64_t M, int64_t N, int64_t K, const float *bias, void *c,
                        int64_t ldc, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  int rc = check_gemm_common(a, b, M, N, K, 128);
  if (rc != FP8_OK) return rc;
  if (sa == nullptr || sb == nullptr) return FP8_ERR_INVALID_ARG;
  if (sfmt != FP8_SCALE_F32 && sfmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
  if ((rc = check_output(c, N, ldc, FP8_OUT_BF16)) != FP8_OK) return rc;
  GemmArgs args{};
  args.M = M; args.N = N; args.K = K; args.fa = FP8_E4M3; args.fb = FP8_E4M3;
  args.out_dt = FP8_OUT_BF16; args.ldc = ldc; args.c = c; args.sa = sa; args.sb = sb;
  args.bias = bias;
  const int mode = sfmt == FP8_SCALE_F32 ? fp8k::kScaleGroupF32 : fp8k::kScaleGroupUe8m0;
  if (g_use_gemv && fp8k::gemv_group_eligible(M, K)) {
    // one row: a stream over the weights on the CUDA cores
    DeviceState *d = nullptr;
    if ((rc = device_state(&d)) != FP8_OK) return rc;
    return to_status(
        fp8k::launch_gemv_group(a, sa, b, sb, sfmt, M, N, K, bias, c, (cudaStream_t)stream));
  }
  if (g_use_skinny && fp8k::gemm_skinny_rows(M) != 0) {
    // 1-128 rows: the weights stream through the few-row kernel (its tile
    // is 128 weight rows x the activation rows padded to 16, 32 or 64; two
    // 64-row halves beyond 64)
    DeviceState *d = nullptr;
    if ((rc = device_state(&d)) != FP8_OK) return rc;
    args.err = d->err;
    args.wait_limit_ns = g_wait_limit_ns;
    args.vec_store = vector_store_ok(c, ldc, FP8_OUT_BF16);
    args.ksplit = fp8k::gemm_skinny_ksplit(M, N, K, d->sms);
    CUtensorMap tmw, tmx;
    if ((rc = encode_operand(&tmw, b, K, N, 128)) != FP8_OK) return rc;
    if ((rc = encode_operand(&tmx, a, K, M, fp8k::gemm_skinny_rows(M))) != FP8_OK) return rc;
    return to_status(fp8k::launch_gemm_skinny(sfmt == FP8_SCALE_F32 ? 0 : 1, tmw, tmx, args,
                                              (cudaStream_t)stream));
  }
  if (mode == fp8k::kScaleGroupUe8m0 && M > 128) {
    // Beyond one row tile: the UE8M0 scales become E8M0 words (four equal
    // bytes per 128-wide K slice) that the block-scaled GEMM bulk-copies per
    // stage, in place of the per-stage byte loads of the group mode.  Same
    // products, same FP32 accumulation: the tensor core applies 2^e to each
    // 1x32 sub-block of the group instead of the group as a whole.  (At
    // K 7168, N 2048 the words measured equal at M = 64-128, slower at
    // M = 16 (the conversion's launch) and faster from M = 256 on.)
    DeviceState *d = nullptr;
    if ((rc = device_state(&d)) != FP8_OK) return rc;
    const size_t G = (size_t)(K / 128);
    const size_t mpad = (size_t)(M + 127) / 128 * 128, npad = (size_t)(N + 127) / 128 * 128;
    void *w = nullptr;
    if ((rc = get_workspace((cudaStream_t)stream, G * (mpad + npad) * 4, &w, kWsWords)) != FP8_OK)
      return rc;
    uint32_t *la = static_cast<uint32_t *>(w), *lb = la + G * mpad;
    if ((rc = to_status(fp8k::launch_ue8m0_words(static_cast<const uint8_t *>(sa),
                                                 static_cast<const uint8_t *>(sb), M, N, K, la, lb,
                                                 d->sms, (cudaStream_t)stream))) != FP8_OK)
      return rc;
    args.sa = la;
    args.sb = lb;
    args.ga = args.gb = nullptr;
    return run_gemm(fp8k::kScaleMx, a, b, args, (cudaStream_t)stream);
  }
  return run_gemm(mode, a, b, args, (cudaStream_t)stream);
}

int fp8_gemm_group_experts(const uint8_t *a, const void *sa, const uint8_t *b, const void *sb,
                           int sfmt, const int32_t *offsets, int experts, int64_t M, int64_t N,
                           int64_t K, void *c, int64_t ldc, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  int rc = check_gemm_common(a, b, M, N, K, 128);
  if (rc != FP8_OK) return rc;
  if (sa == nullptr || sb == nullptr || offsets == nullptr) return FP8_ERR_INVALID_ARG;
  if (experts < 1 || experts > fp8k::kMaxExperts) return FP8_ERR_INVALID_ARG;
  if (experts * N >= kMaxDim) return FP8_ERR_INVALID_ARG;
  if (sfmt != FP8_SCALE_F32 && sfmt != FP8_SCALE_UE8M0) return FP8_ERR_INVALID_ARG;
  if ((rc = check_output(c, N, ldc, FP8_OUT_BF16)) != FP8_OK) return rc;
  DeviceState *d = nullptr;
  if ((rc = device_state(&d)) != FP8_OK) return rc;
  const int mode = sfmt == FP8_SCALE_F32 ? fp8k::kScaleGroupF32 : fp8k::kScaleGroupUe8m0;
  fp8k::GemmArgs args{};
  args.M = M; args.N = N; args.K = K; args.fa = FP8_E4M3; args.fb = FP8_E4M3;
  args.out_dt = FP8_OUT_BF16; args.ldc = ldc; args.c = c; args.sa = sa; args.sb = sb;
  args.err = d->err;
  args.wait_limit_ns = g_wait_limit_ns;
  args.vec_store = vector_store_ok(c, ldc, FP8_OUT_BF16);
  args.ksplit = 1;
  args.experts = experts;
  args.offsets = offsets;
  args.sb_expert_stride = ((N + 127) / 128) * (K / 128);
  // tile width for the expected tile count (about half a row tile of
  // padding per expert)
  CUtensorMap tma, tmb;
  if ((rc = encode_operand(&tma, a, K, M, 128)) != FP8_OK) return rc;
  if (mode == fp8k::kScaleGroupF32 && g_use_pairs &&
      fp8k::gemm_pair_promote_eligible(M, N, K, d->sms)) {
    // FP32 scales on CTA pairs, expert row tiles of 256
    if ((rc = encode_operand(&tmb, b, K, (int64_t)experts * N,
                             fp8k::gemm_pair_promote_b_rows())) != FP8_OK)
      return rc;
    return to_status(fp8k::launch_gemm_pair_promote(tma, tmb, args, d->sms, (cudaStream_t)stream));
  }
  const int bn = fp8k::gemm_tile_n(mode, M + 64 * (int64_t)experts, N, d->sms);
  if ((rc = encode_operand(&tmb, b, K, (int64_t)experts * N, bn)) != FP8_OK) return rc;
  if (mode == fp8k::kScaleGroupUe8m0 && M > 256 && N % 128 == 0) {
    // as in fp8_gemm_group: the UE8M0 scales become E8M0 words for the
    // block-scaled kernel; the A words are stored per expert row tile
    const int64_t G = K / 128, tmax = (M + 127) / 128 + experts;
    const size_t a_words = (size_t)tmax * (size_t)G * 128, b_words = (size_t)G * experts * N;
    void *w = nullptr;
    if ((rc = get_workspace((cudaStream_t)stream, (a_words + b_words) * 4, &w, kWsWords)) != FP8_OK)
      return rc;
    uint32_t *la = static_cast<uint32_t *>(w), *lb = la + a_words;
    if ((rc = to_status(fp8k::launch_ue8m0_words_experts(
             static_cast<const uint8_t *>(sa), static_cast<const uint8_t *>(sb), offsets, experts,
             M, N, K, tmax, la, lb, d->sms, (cudaStream_t)stream))) != FP8_OK)
      return rc;
    args.sa = la;
    args.sb = lb;
    args.ga = args.gb = nullptr;
    return to_status(
        fp8k::launch_gemm_experts(fp8k::kScaleMx, bn, tma, tmb, args, d->sms, (cudaStream_t)stream));
  }
  return to_status(fp8k::launch_gemm_experts(mode, bn, tma, tmb, args, d->sms, (cudaStream_t)stream));
}

int fp8_gemm_mx(const uint8_t *a, const uint32_t *la, const float *ga, const uint8_t *b,
                const uint32_t *lb, const float *gb, int64_t M, int64_t N, int64_t K, int out_dt,
                void *c, int64_t ldc, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  int rc = check_gemm_common(a, b, M, N, K, 128);
  if (rc != FP8_OK) return rc;
  if (la == nullptr || lb == nullptr || ga == nullptr || gb == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned16(la) || !aligned16(lb)) return FP8_ERR_MISALIGNED;
  if ((rc = check_output(c, N, ldc, out_dt)) != FP8_OK) return rc;
  GemmArgs args{};
  args.M = M; args.N = N; args.K = K; args.fa = FP8_E4M3; args.fb = FP8_E4M3;
  args.out_dt = out_dt; args.ldc = ldc; args.c = c; args.sa = la; args.sb = lb;
  args.ga = ga; args.gb = gb;
  return run_gemm(fp8k::kScaleMx, a, b, args, (cudaStream_t)stream);
}

int fp8_gemm_mx_rows(const uint8_t *a, const uint32_t *la, const float *ga, const uint8_t *b,
                     const uint32_t *lb, const float *gb, int64_t M, int64_t N, int64_t K,
                     int out_dt, void *c, int64_t ldc, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  int rc = check_gemm_common(a, b, M, N, K, 128);
  if (rc != FP8_OK) return rc;
  if (la == nullptr || lb == nullptr || ga == nullptr || gb == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned16(la) || !aligned16(lb)) return FP8_ERR_MISALIGNED;
  if ((rc = check_output(c, N, ldc, out_dt)) != FP8_OK) return rc;
  GemmArgs args{};
  args.M = M; args.N = N; args.K = K; args.fa = FP8_E4M3; args.fb = FP8_E4M3;
  args.out_dt = out_dt; args.ldc = ldc; args.c = c; args.sa = la; args.sb = lb;
  args.ga = ga; args.gb = gb;
  args.row_scale = ga;  // S_a[m] * S_b[n] per output element, in the epilogue
  args.col_scale = gb;
  return run_gemm(fp8k::kScaleMx, a, b, args, (cudaStream_t)stream);
}

int fp8_delayed_state_update(float *hist, float *scale, const float *amax_cur, int64_t L,
                             int fmt, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (hist == nullptr || scale == nullptr || amax_cur == nullptr || !valid_fmt(fmt))
    return FP8_ERR_INVALID_ARG;
  if (L < 1 || L > 32768) return FP8_ERR_INVALID_ARG;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_delayed_update(hist, scale, amax_cur, L, fmt, (cudaStream_t)stream));
}

int fp8_delayed_state_update_multi(const fp8_delayed_item_t *items, int count,
                                   fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (items == nullptr || count < 1 || count > fp8k::kMaxDelayed) return FP8_ERR_INVALID_ARG;
  fp8k::DelayedItems it{};
  for (int i = 0; i < count; ++i) {
    const fp8_delayed_item_t &d = items[i];
    if (d.hist == nullptr || d.scale == nullptr || d.amax_cur == nullptr || !valid_fmt(d.fmt))
      return FP8_ERR_INVALID_ARG;
    if (d.L < 1 || d.L > 32768) return FP8_ERR_INVALID_ARG;
    // no two items write the same memory (their updates run concurrently)
    for (int j = 0; j < i; ++j) {
      const fp8_delayed_item_t &e = items[j];
      const bool hist_overlap = d.hist < e.hist + e.L && e.hist < d.hist + d.L;
      const bool scale_in_hist = (d.scale >= e.hist && d.scale < e.hist + e.L) ||
                                 (e.scale >= d.hist && e.scale < d.hist + d.L);
      if (hist_overlap || scale_in_hist || d.scale == e.scale) return FP8_ERR_INVALID_ARG;
    }
    if (d.scale >= d.hist && d.scale < d.hist + d.L) return FP8_ERR_INVALID_ARG;
    it.hist[i] = d.hist;
    it.scale[i] = d.scale;
    it.amax_cur[i] = d.amax_cur;
    it.L[i] = d.L;
    it.fmt[i] = d.fmt;
  }
  it.count = count;
  DeviceState *dev = nullptr;
  int rc = device_state(&dev);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_delayed_update_multi(it, (cudaStream_t)stream));
}

int fp8_auto_weight_scale(const float *amax0, int64_t t, double lr, int fmt, float *scale_out,
                          fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (amax0 == nullptr || scale_out == nullptr || t < 0 || !valid_fmt(fmt) || !(lr >= 0.0))
    return FP8_ERR_INVALID_ARG;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_auto_scale(amax0, lr * (double)t, fmt, scale_out,
                                           (cudaStream_t)stream));
}

int fp8_swiglu_forward(const void *h, const void *u, void *a, int64_t n, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (n < 0 || (n > 0 && (h == nullptr || u == nullptr || a == nullptr)))
    return FP8_ERR_INVALID_ARG;
  if (n % 8 != 0 || !aligned16(h) || !aligned16(u) || !aligned16(a)) return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  if (n == 0) return FP8_OK;
  return to_status(fp8k::launch_swiglu_fwd(h, u, a, n, d->sms, (cudaStream_t)stream));
}

int fp8_swiglu_backward(const void *da, const void *h, const void *u, void *dh, void *du,
                        int64_t n, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (n < 0 || (n > 0 && (da == nullptr || h == nullptr || u == nullptr || dh == nullptr ||
                          du == nullptr)))
    return FP8_ERR_INVALID_ARG;
  if (n % 8 != 0 || !aligned16(da) || !aligned16(h) || !aligned16(u) || !aligned16(dh) ||
      !aligned16(du))
    return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  if (n == 0) return FP8_OK;
  return to_status(fp8k::launch_swiglu_bwd(da, h, u, dh, du, n, d->sms, (cudaStream_t)stream));
}

int fp8_swiglu_forward_quantize(const void *h, const void *u, int64_t n, int fmt,
                                const float *scale, uint8_t *q, float *amax_out,
                                fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (n < 0 || !valid_fmt(fmt)) return FP8_ERR_INVALID_ARG;
  // an empty tensor is read and written nowhere: its pointers may be null
  if (n > 0 && (h == nullptr || u == nullptr || scale == nullptr || q == nullptr))
    return FP8_ERR_INVALID_ARG;
  if (amax_out != nullptr && amax_out == scale) return FP8_ERR_INVALID_ARG;
  if (n % 8 != 0 || !aligned16(h) || !aligned16(u) || !aligned16(q)) return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_swiglu_fwd_quant(h, u, n, fmt, scale, q, amax_out, d->sms,
                                                 (cudaStream_t)stream));
}

int fp8_swiglu_backward_quantize(const void *da, const void *h, const void *u, int64_t n, int fmt,
                                 const float *scale_dh, const float *scale_du, uint8_t *q_dh,
                                 uint8_t *q_du, float *amax_dh, float *amax_du,
                                 fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (n < 0 || !valid_fmt(fmt)) return FP8_ERR_INVALID_ARG;
  if (n > 0 && (da == nullptr || h == nullptr || u == nullptr || scale_dh == nullptr ||
                scale_du == nullptr || q_dh == nullptr || q_du == nullptr))
    return FP8_ERR_INVALID_ARG;
  if ((amax_dh == nullptr) != (amax_du == nullptr)) return FP8_ERR_INVALID_ARG;
  if (amax_dh != nullptr &&
      (amax_dh == amax_du || amax_dh == scale_dh || amax_dh == scale_du ||
       amax_du == scale_dh || amax_du == scale_du))
    return FP8_ERR_INVALID_ARG;
  if (n % 8 != 0 || !aligned16(da) || !aligned16(h) || !aligned16(u) || !aligned16(q_dh) ||
      !aligned16(q_du))
    return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_swiglu_bwd_quant(da, h, u, n, fmt, scale_dh, scale_du, q_dh, q_du,
                                                 amax_dh, amax_du, d->sms, (cudaStream_t)stream));
}

int fp8_adamw_multi(const fp8_adamw_item_t *items, int count, int64_t *step, int advance,
                    double lr, double beta1, double beta2, double eps, double weight_decay,
                    fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (step == nullptr || count < 0 || count > fp8k::kMaxAdamw || (count > 0 && items == nullptr))
    return FP8_ERR_INVALID_ARG;
  if (advance != 0 && advance != 1) return FP8_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(step) & 7u) != 0) return FP8_ERR_MISALIGNED;
  fp8k::AdamwMulti a{};
  for (int k = 0; k < count; ++k) {
    const fp8_adamw_item_t &it = items[k];
    if (it.n < 0 || (it.n > 0 && (it.p == nullptr || it.g == nullptr || it.m == nullptr ||
                                  it.v == nullptr)))
      return FP8_ERR_INVALID_ARG;
    if (it.n % 4 != 0) return FP8_ERR_MISALIGNED;
    if (it.n > 0 && (!aligned16(it.p) || !aligned16(it.g) || !aligned16(it.m) ||
                     !aligned16(it.v) ||
                     (it.p_bf16 != nullptr && (reinterpret_cast<uintptr_t>(it.p_bf16) & 7u) != 0)))
      return FP8_ERR_MISALIGNED;
    if (it.q != nullptr) {
      if (it.q_scale == nullptr || !valid_fmt(it.q_fmt)) return FP8_ERR_INVALID_ARG;
      if (it.q_amax != nullptr && reinterpret_cast<const void *>(it.q_amax) ==
                                      reinterpret_cast<const void *>(it.q_scale))
        return FP8_ERR_INVALID_ARG;
      for (int j = 0; j < k; ++j)
        if (it.q_amax != nullptr && items[j].q != nullptr && items[j].q_amax == it.q_amax)
          return FP8_ERR_INVALID_ARG;
      if ((reinterpret_cast<uintptr_t>(it.q) & 3u) != 0) return FP8_ERR_MISALIGNED;
      a.q[k] = it.q;
      a.q_scale[k] = it.q_scale;
      a.q_amax[k] = reinterpret_cast<uint32_t *>(it.q_amax);
      a.q_fmt[k] = it.q_fmt;
    }
    a.p[k] = it.p;
    a.g[k] = it.g;
    a.m[k] = it.m;
    a.v[k] = it.v;
    a.pb[k] = it.p_bf16;
    a.n[k] = it.n;
  }
  a.count = count;
  a.step = step;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  return to_status(fp8k::launch_adamw_multi(a, advance != 0, lr, beta1, beta2, eps, weight_decay,
                                            d->sms, (cudaStream_t)stream));
}

int fp8_adamw_step(float *p, const float *g, float *m, float *v, void *p_bf16, int64_t n,
                   int64_t step, double lr, double beta1, double beta2, double eps,
                   double weight_decay, fp8_stream_t stream) {
  const NvtxRange nvtx_range(__func__);
  if (p == nullptr || g == nullptr || m == nullptr || v == nullptr || n < 0 || step < 1)
    return FP8_ERR_INVALID_ARG;
  if (n % 4 != 0 || !aligned16(p) || !aligned16(g) || !aligned16(m) || !aligned16(v) ||
      (p_bf16 != nullptr && (reinterpret_cast<uintptr_t>(p_bf16) & 7u) != 0))
    return FP8_ERR_MISALIGNED;
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  if (n == 0) return FP8_OK;
  return to_status(fp8k::launch_adamw(p, g, m, v, p_bf16, n, step, lr, beta1, beta2, eps,
                                      weight_decay, d->sms, (cudaStream_t)stream));
}

const char *fp8_status_string(int status) {
  switch (status) {
    case FP8_OK: return "ok";
    case FP8_ERR_INVALID_ARG: return "invalid argument";
    case FP8_ERR_MISALIGNED: return "misaligned pointer, stride or K granularity";
    case FP8_ERR_UNSUPPORTED: return "unsupported format combination or shape";
    case FP8_ERR_CUDA: return "CUDA runtime error";
    case FP8_ERR_TIMEOUT: return "device-side wait timed out";
    case FP8_ERR_NO_DEVICE: return "no sm_103 device is current";
    case FP8_ERR_SCRATCH_LIMIT: return "shape exceeds the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

int fp8_get_last_device_error(int *where_out, fp8_stream_t stream) {
  DeviceState *d = nullptr;
  int rc = device_state(&d);
  if (rc != FP8_OK) return rc;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return FP8_ERR_CUDA;
  uint32_t h[2] = {0, 0};
  if (cudaMemcpy(h, d->err, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FP8_ERR_CUDA;
  if (h[0] != 0) {
    const uint32_t z[2] = {0, 0};
    if (cudaMemcpy(d->err, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return FP8_ERR_CUDA;
  }
  if (where_out != nullptr) *where_out = (int)h[1];
  return -(int)h[0];
}

int fp8_set_option(int option, int value) {
  if (option == FP8_OPT_GEMM_CTA_PAIRS) {
    g_use_pairs = value != 0;
    return FP8_OK;
  }
  if (option == FP8_OPT_GEMM_FEW_ROWS) {
    g_use_gemv = value != 0;
    return FP8_OK;
  }
  if (option == FP8_OPT_GEMM_SKINNY) {
    g_use_skinny = value != 0;
    return FP8_OK;
  }
  if (option == FP8_OPT_GEMM_TMA_STORE) {
    g_use_tma_store = value != 0;
    return FP8_OK;
  }
  if (option == FP8_OPT_GEMM_MULTICAST) {
    g_use_multicast = value != 0;
    return FP8_OK;
  }
  if (option == FP8_OPT_GEMM_BAND_ROWS) {
    if (value < 1 || value > 4096) return FP8_ERR_INVALID_ARG;
    g_pair_band_rows = value;
    return FP8_OK;
  }
  if (option == FP8_OPT_WAIT_LIMIT_US) {
    if (value < 0) return FP8_ERR_INVALID_ARG;
    g_wait_limit_ns = (uint64_t)value * 1000ull;
    return FP8_OK;
  }
  return FP8_ERR_INVALID_ARG;
}

const char *fp8_version(void) { return "fp8gemm 0.1 (sm_103a)"; }

}  // extern "C"
