// Split-K BF16 GEMM for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory for a workspace: code
// running inside a host framework whose allocator owns the whole device
// pool and forbids foreign allocations, serving loops that must not call the
// CUDA allocator once warmed up (an allocation can synchronise the device
// and stall every stream), and plugins that are handed raw pointers but no
// allocator.  gemm_bf16_nt_splitk_static gives them split-K without a
// workspace argument: the FP32 partial tiles live in a fixed-size scratch
// array that is part of this library's device image.
//
// The array is a file-scope __device__ variable.  In host code its name only
// stands in for the symbol (it is not a device address), so the address is
// looked up once per device with cudaGetSymbolAddress, with that device
// current, during the library's per-device set-up (the first call of any
// entry point on that device), and that pointer is what the kernels
// receive.  Every GPU that loads the library holds the array until the
// process exits.
#include <cstdint>

#include "internal.h"

static_assert(GEMM_SPLITK_STATIC_SCRATCH_BYTES % 256 == 0, "scratch size");
static __device__ __align__(256) float g_splitk_scratch[GEMM_SPLITK_STATIC_SCRATCH_BYTES / 4];

namespace gb300 {

// Called once per device, with that device current, by the library's
// per-device set-up (current_device): the scratch array's device address.
int splitk_static_scratch_lookup(float** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_splitk_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return GEMM_ERR_NO_DEVICE;
  }
  *out = static_cast<float*>(p);
  return GEMM_OK;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" int gemm_bf16_nt_splitk_static(const void* A, const void* B, void* C, int M, int N,
                                          int K, int k_splits, void* stream) {
  if (!A || !B || !C) return GEMM_ERR_NULL;
  if (M <= 0 || N <= 0 || K <= 0 || k_splits < 1 || k_splits > 64) return GEMM_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return GEMM_ERR_ALIGN;
  if (K % 8 != 0 || N % 8 != 0) return GEMM_ERR_ALIGN;
  int kbps = 0;
  const int splits = splitk_effective_splits(K, k_splits, &kbps);
  const size_t need = size_t(splits) * size_t(M) * size_t(N) * 4;
  if (need > GEMM_SPLITK_STATIC_SCRATCH_BYTES) return GEMM_ERR_SHAPE;  // beyond the fixed scratch
  const size_t sc = size_t(M) * N * 2;
  if (overlaps(C, sc, A, size_t(M) * K * 2) || overlaps(C, sc, B, size_t(N) * K * 2))
    return GEMM_ERR_ALIAS;
  DeviceInfo dev;
  const int rc = current_device(&dev, stream);  // set-up looks up dev.splitk_scratch
  if (rc != GEMM_OK) return rc;
  // Every element of the scratch that the reduce reads is written earlier in
  // this same call, so nothing needs clearing between calls.
  return launch_gemm_bf16_splitk(A, B, C, dev.splitk_scratch, M, N, K, k_splits, dev,
                                 static_cast<cudaStream_t>(stream));
}
