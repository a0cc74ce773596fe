// C ABI of the library (declared in include/gb300gemm.h): argument
// validation, per-device state (SM count, status word), TMA descriptor
// encoding, dispatch to the launchers.  Validation is pure host code and
// runs before any CUDA call, so a bad call never touches the device.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "internal.h"

namespace gb300 {

// Device status word: 0, or 0x100 | where for the first bounded wait that
// ran out since it was last cleared.
__device__ unsigned int g_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceSlot {
  bool ready = false;
  int rc = GEMM_OK;
  DeviceInfo info{};
};

std::mutex g_dev_mutex;
DeviceSlot g_devices[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a+na) and [b, b+nb) overlap?
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

constexpr long long kMaxTiles = 1ll << 30;

}  // namespace

int current_device(DeviceInfo* out, void* stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  // A host thread that has made no CUDA runtime call of its own has no
  // current context, and the driver's tensor-map encoder needs one: then
  // make the device's primary context current in this thread.  A context
  // the caller made current (primary or not) is left as it is.
  {
    CtxGetCurrentFn get = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    const CUresult r = get ? get(&ctx) : CUDA_ERROR_NOT_INITIALIZED;
    if ((r != CUDA_SUCCESS || ctx == nullptr) && cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_NO_DEVICE;
    }
  }
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceSlot& s = g_devices[dev];
  if (!s.ready) {
    // One-time set-up of this device: attributes and the device addresses of
    // the library's __device__ variables.  Symbol lookups may load the
    // module, which a stream capture does not allow: refuse during capture
    // and leave the set-up for a later call.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap) != cudaSuccess ||
        cap != cudaStreamCaptureStatusNone) {
      cudaGetLastError();
      return GEMM_ERR_CAPTURE;
    }
    DeviceInfo d{};
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_NO_DEVICE;  // not cached: a later call retries
    }
    int rc = GEMM_OK;
    if (!(d.cc_major == 10 && d.cc_minor == 3)) {
      rc = GEMM_ERR_ARCH;  // the library carries sm_103a code only
    } else if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word) !=
                   cudaSuccess ||
               splitk_static_scratch_lookup(&d.splitk_scratch) != GEMM_OK) {
      cudaGetLastError();
      return GEMM_ERR_NO_DEVICE;  // not cached: a later call retries
    }
    s.info = d;
    s.rc = rc;  // GEMM_OK, or the permanent GEMM_ERR_ARCH
    s.ready = true;
  }
  *out = s.info;
  return s.rc;
}

unsigned long long wait_timeout_ns() { return 2000ull * 1000000ull; }

namespace {
// Testing overrides (gemm_testing_set_overrides); 0 = the shape decides.
std::atomic<int> g_test_cta_group{0};
std::atomic<int> g_test_streamk_clusters{0};
}  // namespace

int testing_cta_group() { return g_test_cta_group.load(std::memory_order_relaxed); }
int testing_streamk_clusters() { return g_test_streamk_clusters.load(std::memory_order_relaxed); }

int encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base,
                   uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1,
                   CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return GEMM_ERR_NO_DEVICE;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * uint64_t(elem_bytes), d0 * d1 * uint64_t(elem_bytes)};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_LAUNCH;
}

int encode_tmap_3d_strided(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                           uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                           uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2,
                           CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return GEMM_ERR_NO_DEVICE;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_LAUNCH;
}

namespace {

// Shared checks of the BF16 NT family.
int check_bf16_nt(const void* A, const void* B, const void* C, int M, int N, int K,
                  size_t c_elem_bytes) {
  if (!A || !B || !C) return GEMM_ERR_NULL;
  if (M <= 0 || N <= 0 || K <= 0) return GEMM_ERR_SHAPE;
  const long long tiles = (long long)((M + 127) / 128) * ((N + 63) / 64);
  if (tiles > kMaxTiles) return GEMM_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return GEMM_ERR_ALIGN;
  if (K % 8 != 0) return GEMM_ERR_ALIGN;  // 16-byte row pitch of A and B
  const size_t sa = size_t(M) * K * 2, sb = size_t(N) * K * 2, sc = size_t(M) * N * c_elem_bytes;
  if (overlaps(C, sc, A, sa) || overlaps(C, sc, B, sb)) return GEMM_ERR_ALIAS;
  return GEMM_OK;
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" {

int gemm_bf16_nt(const void* A, const void* B, void* C, int M, int N, int K, void* stream) {
  int rc = check_bf16_nt(A, B, C, M, N, K, 2);
  if (rc != GEMM_OK) return rc;
  if (N % 8 != 0) return GEMM_ERR_ALIGN;  // 16-byte row pitch of C
  DeviceInfo dev;
  if ((rc = current_device(&dev, stream)) != GEMM_OK) return rc;
  return launch_gemm_bf16(A, B, C, M, N, K, 0.0f, false, dev, static_cast<cudaStream_t>(stream));
}

int gemm_bf16_nn(const void* A, const void* B, void* C, int M, int N, int K, void* stream) {
  if (!A || !B || !C) return GEMM_ERR_NULL;
  if (M <= 0 || N <= 0 || K <= 0) return GEMM_ERR_SHAPE;
  const long long tiles = (long long)((M + 127) / 128) * ((N + 63) / 64);
  if (tiles > kMaxTiles) return GEMM_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return GEMM_ERR_ALIGN;
  if (K % 8 != 0 || N % 8 != 0) return GEMM_ERR_ALIGN;  // 16-byte row pitch of A, B and C
  const size_t sa = size_t(M) * K * 2, sb = size_t(K) * N * 2, sc = size_t(M) * N * 2;
  if (overlaps(C, sc, A, sa) || overlaps(C, sc, B, sb)) return GEMM_ERR_ALIAS;
  DeviceInfo dev;
  int rc = current_device(&dev, stream);
  if (rc != GEMM_OK) return rc;
  return launch_gemm_bf16_nn(A, B, C, M, N, K, dev, static_cast<cudaStream_t>(stream));
}

int gemm_bf16_nt_scaled_acc(const void* A, const void* B, void* C_inout, int M, int N, int K,
                            float scale, void* stream) {
  int rc = check_bf16_nt(A, B, C_inout, M, N, K, 2);
  if (rc != GEMM_OK) return rc;
  if (N % 8 != 0) return GEMM_ERR_ALIGN;
  DeviceInfo dev;
  if ((rc = current_device(&dev, stream)) != GEMM_OK) return rc;
  return launch_gemm_bf16(A, B, C_inout, M, N, K, scale, true, dev,
                          static_cast<cudaStream_t>(stream));
}

int gemm_bf16_nt_splitk(const void* A, const void* B, void* C, void* workspace,
                        size_t workspace_bytes, int M, int N, int K, int k_splits, void* stream) {
  int rc = check_bf16_nt(A, B, C, M, N, K, 2);
  if (rc != GEMM_OK) return rc;
  if (N % 8 != 0) return GEMM_ERR_ALIGN;
  if (!workspace) return GEMM_ERR_NULL;
  if (k_splits < 1 || k_splits > 64) return GEMM_ERR_SHAPE;
  if (!aligned16(workspace)) return GEMM_ERR_ALIGN;
  int kbps = 0;
  const int s_eff = splitk_effective_splits(K, k_splits, &kbps);
  const size_t need = size_t(s_eff) * size_t(M) * size_t(N) * 4;
  if (workspace_bytes < need) return GEMM_ERR_SHAPE;
  const size_t sa = size_t(M) * K * 2, sb = size_t(N) * K * 2, sc = size_t(M) * N * 2;
  if (overlaps(workspace, need, A, sa) || overlaps(workspace, need, B, sb) ||
      overlaps(workspace, need, C, sc))
    return GEMM_ERR_ALIAS;
  DeviceInfo dev;
  if ((rc = current_device(&dev, stream)) != GEMM_OK) return rc;
  return launch_gemm_bf16_splitk(A, B, C, static_cast<float*>(workspace), M, N, K, k_splits, dev,
                                 static_cast<cudaStream_t>(stream));
}

size_t gemm_bf16_nt_splitk_workspace_bytes(int M, int N, int K, int k_splits) {
  if (M <= 0 || N <= 0 || K <= 0 || k_splits < 1 || k_splits > 64) return 0;
  int kbps = 0;
  const int s_eff = splitk_effective_splits(K, k_splits, &kbps);
  return size_t(s_eff) * size_t(M) * size_t(N) * 4;
}

int gemm_bf16_nt_streamk(const void* A, const void* B, void* C, void* workspace,
                         size_t workspace_bytes, int M, int N, int K, void* stream) {
  int rc = check_bf16_nt(A, B, C, M, N, K, 2);
  if (rc != GEMM_OK) return rc;
  if (N % 8 != 0) return GEMM_ERR_ALIGN;
  if (!workspace) return GEMM_ERR_NULL;
  if (!aligned16(workspace)) return GEMM_ERR_ALIGN;
  // the whole buffer the caller hands over must be disjoint from the matrices
  const size_t sa = size_t(M) * K * 2, sb = size_t(N) * K * 2, sc = size_t(M) * N * 2;
  if (overlaps(workspace, workspace_bytes, A, sa) || overlaps(workspace, workspace_bytes, B, sb) ||
      overlaps(workspace, workspace_bytes, C, sc))
    return GEMM_ERR_ALIAS;
  DeviceInfo dev;
  if ((rc = current_device(&dev, stream)) != GEMM_OK) return rc;
  if (workspace_bytes < streamk_workspace_bytes(dev)) return GEMM_ERR_SHAPE;
  return launch_gemm_bf16_streamk(A, B, C, static_cast<float*>(workspace), M, N, K, dev,
                                  static_cast<cudaStream_t>(stream));
}

size_t gemm_bf16_nt_streamk_workspace_bytes(void) {
  DeviceInfo dev;
  if (current_device(&dev, nullptr) != GEMM_OK) return 0;
  return streamk_workspace_bytes(dev);
}

int gemm_w4a16(const void* A, const void* b, const void* sfb, float scale2, void* C, int M, int N,
               int K, void* stream) {
  if (!A || !b || !sfb || !C) return GEMM_ERR_NULL;
  if (M <= 0 || N <= 0 || K <= 0) return GEMM_ERR_SHAPE;
  const long long tiles = (long long)((M + 255) / 256) * ((N + 255) / 256);
  if (tiles > kMaxTiles) return GEMM_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(b) || !aligned16(sfb) || !aligned16(C)) return GEMM_ERR_ALIGN;
  if (K % 256 != 0 || N % 8 != 0) return GEMM_ERR_ALIGN;  // 16-byte rows of sfb, b and C
  const size_t sa = size_t(M) * K * 2, sbq = size_t(N) * (K / 2), ss = size_t(N) * (K / 16);
  const size_t sc = size_t(M) * N * 2;
  if (overlaps(C, sc, A, sa) || overlaps(C, sc, b, sbq) || overlaps(C, sc, sfb, ss))
    return GEMM_ERR_ALIAS;
  DeviceInfo dev;
  int rc = current_device(&dev, stream);
  if (rc != GEMM_OK) return rc;
  return launch_gemm_w4a16(A, static_cast<const uint8_t*>(b), static_cast<const uint8_t*>(sfb),
                           scale2, C, M, N, K, dev, static_cast<cudaStream_t>(stream));
}

int gemm_w4a16_t(const void* A, const void* b_t, const void* sfb_t, float scale2, void* C, int M,
                 int N, int K, int ldb, void* stream) {
  if (!A || !b_t || !sfb_t || !C) return GEMM_ERR_NULL;
  if (M <= 0 || N <= 0 || K <= 0 || ldb < N) return GEMM_ERR_SHAPE;
  const long long tiles = (long long)((M + 255) / 256) * ((N + 255) / 256);
  if (tiles > kMaxTiles) return GEMM_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(b_t) || !aligned16(sfb_t) || !aligned16(C))
    return GEMM_ERR_ALIGN;
  if (K % 128 != 0 || ldb % 16 != 0) return GEMM_ERR_ALIGN;  // whole K blocks; 16-byte rows
  const size_t sa = size_t(M) * K * 2, sbq = size_t(K / 2) * ldb, ss = size_t(K / 16) * ldb;
  const size_t sc = size_t(M) * N * 2;
  if (overlaps(C, sc, A, sa) || overlaps(C, sc, b_t, sbq) || overlaps(C, sc, sfb_t, ss))
    return GEMM_ERR_ALIAS;
  DeviceInfo dev;
  int rc = current_device(&dev, stream);
  if (rc != GEMM_OK) return rc;
  return launch_gemm_w4a16_t(A, static_cast<const uint8_t*>(b_t),
                             static_cast<const uint8_t*>(sfb_t), scale2, C, M, N, K, ldb, dev,
                             static_cast<cudaStream_t>(stream));
}

int gemm_w4a16_ws(const void* A, const void* b, const void* sfb, float scale2, void* C,
                  void* workspace, size_t workspace_bytes, int M, int N, int K, void* stream) {
  if (!A || !b || !sfb || !C || !workspace) return GEMM_ERR_NULL;
  if (M <= 0 || N <= 0 || K <= 0) return GEMM_ERR_SHAPE;
  const long long tiles = (long long)((M + 255) / 256) * ((N + 255) / 256);
  if (tiles > kMaxTiles) return GEMM_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(b) || !aligned16(sfb) || !aligned16(C) || !aligned16(workspace))
    return GEMM_ERR_ALIGN;
  if (K % 256 != 0 || N % 8 != 0) return GEMM_ERR_ALIGN;
  const size_t need = size_t(N) * size_t(K) * 2;
  if (workspace_bytes < need) return GEMM_ERR_SHAPE;
  const size_t sa = size_t(M) * K * 2, sbq = size_t(N) * (K / 2), ss = size_t(N) * (K / 16);
  const size_t sc = size_t(M) * N * 2;
  if (overlaps(C, sc, A, sa) || overlaps(C, sc, b, sbq) || overlaps(C, sc, sfb, ss) ||
      overlaps(workspace, need, A, sa) || overlaps(workspace, need, b, sbq) ||
      overlaps(workspace, need, sfb, ss) || overlaps(workspace, need, C, sc))
    return GEMM_ERR_ALIAS;
  DeviceInfo dev;
  int rc = current_device(&dev, stream);
  if (rc != GEMM_OK) return rc;
  return launch_gemm_w4a16_twopass(A, static_cast<const uint8_t*>(b),
                                   static_cast<const uint8_t*>(sfb), scale2, C,
                                   static_cast<uint16_t*>(workspace), M, N, K, dev,
                                   static_cast<cudaStream_t>(stream));
}

size_t gemm_w4a16_ws_workspace_bytes(int N, int K) {
  if (N <= 0 || K <= 0 || K % 256 != 0) return 0;
  return size_t(N) * size_t(K) * 2;
}

int gemm_bf16_nt_ordered(const void* A, const void* B, float* C, int M, int N, int K,
                         void* stream) {
  int rc = check_bf16_nt(A, B, C, M, N, K, 4);
  if (rc != GEMM_OK) return rc;
  DeviceInfo dev;
  if ((rc = current_device(&dev, stream)) != GEMM_OK) return rc;
  return launch_gemm_router(A, B, C, M, N, K, dev, static_cast<cudaStream_t>(stream));
}

int gemm_nvfp4_bs(const void* a, const void* b, const void* sfa, const void* sfb, void* c, int L,
                  int M, int N, int K, void* stream) {
  if (!a || !b || !sfa || !sfb || !c) return GEMM_ERR_NULL;
  if (L <= 0 || M <= 0 || N <= 0 || K <= 0) return GEMM_ERR_SHAPE;
  if (M % 128 != 0 || N % 128 != 0 || K % 256 != 0) return GEMM_ERR_SHAPE;
  const long long tiles = (long long)L * (M / 128) * ((N + 255) / 256);
  if (tiles > kMaxTiles) return GEMM_ERR_SHAPE;
  if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb) || !aligned16(c))
    return GEMM_ERR_ALIGN;
  const size_t sa = size_t(L) * M * (K / 2), sb = size_t(L) * N * (K / 2);
  const size_t ssa = size_t(L) * M * (K / 16), ssb = size_t(L) * N * (K / 16);
  const size_t sc = size_t(L) * M * N * 2;
  if (overlaps(c, sc, a, sa) || overlaps(c, sc, b, sb) || overlaps(c, sc, sfa, ssa) ||
      overlaps(c, sc, sfb, ssb))
    return GEMM_ERR_ALIAS;
  DeviceInfo dev;
  int rc = current_device(&dev, stream);
  if (rc != GEMM_OK) return rc;
  return launch_gemm_nvfp4(a, b, sfa, sfb, c, L, M, N, K, dev, static_cast<cudaStream_t>(stream));
}

size_t gemm_nvfp4_bs_splitk_workspace_bytes(int M, int N, int K, int k_splits) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 256 != 0 || k_splits < 1 || k_splits > 64) return 0;
  int kbps = 0;
  const int s_eff = nvfp4_splitk_effective_splits(K, k_splits, &kbps);
  return size_t(s_eff) * size_t(M) * size_t(N) * 4;
}

int gemm_nvfp4_bs_splitk(const void* a, const void* b, const void* sfa, const void* sfb, void* c,
                         void* workspace, size_t workspace_bytes, int L, int M, int N, int K,
                         int k_splits, void* stream) {
  if (!a || !b || !sfa || !sfb || !c || !workspace) return GEMM_ERR_NULL;
  if (L <= 0 || M <= 0 || N <= 0 || K <= 0) return GEMM_ERR_SHAPE;
  if (M % 128 != 0 || N % 128 != 0 || K % 256 != 0) return GEMM_ERR_SHAPE;
  if (k_splits < 1 || k_splits > 64) return GEMM_ERR_SHAPE;
  int kbps = 0;
  const int s_eff = nvfp4_splitk_effective_splits(K, k_splits, &kbps);
  const long long units = (long long)s_eff * L * ((M + 255) / 256) * ((N + 255) / 256);
  if (units > kMaxTiles) return GEMM_ERR_SHAPE;
  const size_t need = size_t(s_eff) * size_t(L) * size_t(M) * size_t(N) * 4;
  if (workspace_bytes < need) return GEMM_ERR_SHAPE;
  if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb) || !aligned16(c) ||
      !aligned16(workspace))
    return GEMM_ERR_ALIGN;
  const size_t sa = size_t(L) * M * (K / 2), sb = size_t(L) * N * (K / 2);
  const size_t ssa = size_t(L) * M * (K / 16), ssb = size_t(L) * N * (K / 16);
  const size_t sc = size_t(L) * M * N * 2;
  if (overlaps(c, sc, a, sa) || overlaps(c, sc, b, sb) || overlaps(c, sc, sfa, ssa) ||
      overlaps(c, sc, sfb, ssb))
    return GEMM_ERR_ALIAS;
  if (overlaps(workspace, need, a, sa) || overlaps(workspace, need, b, sb) ||
      overlaps(workspace, need, sfa, ssa) || overlaps(workspace, need, sfb, ssb) ||
      overlaps(workspace, need, c, sc))
    return GEMM_ERR_ALIAS;
  DeviceInfo dev;
  int rc = current_device(&dev, stream);
  if (rc != GEMM_OK) return rc;
  return launch_gemm_nvfp4_splitk(a, b, sfa, sfb, c, static_cast<float*>(workspace), L, M, N, K,
                                  k_splits, dev, static_cast<cudaStream_t>(stream));
}

int bf16_scaled_add(void* out, const void* d, float scale, long n, void* stream) {
  if (!out || !d) return GEMM_ERR_NULL;
  if (n <= 0) return GEMM_ERR_SHAPE;
  if (!aligned16(out) || !aligned16(d)) return GEMM_ERR_ALIGN;
  if (overlaps(out, size_t(n) * 2, d, size_t(n) * 2)) return GEMM_ERR_ALIAS;
  DeviceInfo dev;
  int rc = current_device(&dev, stream);
  if (rc != GEMM_OK) return rc;
  return launch_scaled_add(out, d, scale, n, dev, static_cast<cudaStream_t>(stream));
}

int gemm_get_device_status(void* stream) {
  DeviceInfo dev;
  int rc = current_device(&dev, stream);
  if (rc != GEMM_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  unsigned int v = 0;
  if (cudaMemcpy(&v, dev.status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GEMM_ERR_LAUNCH;
  if (v != 0) {
    const unsigned int zero = 0;
    cudaMemcpy(dev.status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    return GEMM_ERR_TIMEOUT;
  }
  return GEMM_OK;
}

int gemm_testing_set_overrides(int cta_group, int streamk_clusters) {
  if (cta_group != 0 && cta_group != 1 && cta_group != 2) return GEMM_ERR_SHAPE;
  if (streamk_clusters < 0) return GEMM_ERR_SHAPE;
  g_test_cta_group.store(cta_group, std::memory_order_relaxed);
  g_test_streamk_clusters.store(streamk_clusters, std::memory_order_relaxed);
  return GEMM_OK;
}

int gemm_selftest_wait_timeout(int timeout_ms, void* stream) {
  if (timeout_ms < 1 || timeout_ms > 10000) return GEMM_ERR_SHAPE;
  DeviceInfo dev;
  int rc = current_device(&dev, stream);
  if (rc != GEMM_OK) return rc;
  return launch_selftest_timeout(timeout_ms, dev, static_cast<cudaStream_t>(stream));
}

const char* gemm_status_string(int status) {
  switch (status) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_NULL: return "GEMM_ERR_NULL: a required pointer is NULL";
    case GEMM_ERR_SHAPE: return "GEMM_ERR_SHAPE: invalid dimensions";
    case GEMM_ERR_ALIGN: return "GEMM_ERR_ALIGN: pointer or row pitch not 16-byte aligned";
    case GEMM_ERR_ALIAS: return "GEMM_ERR_ALIAS: output overlaps an input";
    case GEMM_ERR_ARCH: return "GEMM_ERR_ARCH: device is not sm_103";
    case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: a CUDA call failed";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a kernel ran out of a bounded wait";
    case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE: no usable CUDA device";
    case GEMM_ERR_CAPTURE:
      return "GEMM_ERR_CAPTURE: first call on this device made during stream capture";
    default: return "unknown status";
  }
}

}  // extern "C"
