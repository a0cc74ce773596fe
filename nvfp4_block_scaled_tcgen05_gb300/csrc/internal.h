// Declarations shared by the host-side translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gb300gemm.h"

namespace gb300 {

// Per-device facts the launchers need; filled once per device.
struct DeviceInfo {
  int device;
  int num_sms;
  int cc_major, cc_minor;
  unsigned int* status;   // device address of the status word
  float* splitk_scratch;  // device address of the allocation-free split-K scratch
};

// Fills `out` for the current device; the first call per device does the
// one-time set-up (attributes, device addresses of the library's __device__
// variables), which cannot run while `stream` is being captured.  Returns
// GEMM_OK, GEMM_ERR_NO_DEVICE, GEMM_ERR_ARCH (not an sm_103 GPU) or
// GEMM_ERR_CAPTURE (set-up still due and `stream` is capturing).
int current_device(DeviceInfo* out, void* stream);

// Device address of the allocation-free split-K scratch array on the
// current device (splitk_static.cu); called by the per-device set-up.
// Returns GEMM_OK or GEMM_ERR_NO_DEVICE.
int splitk_static_scratch_lookup(float** out);

// Bound on every device-side wait, in nanoseconds (2 s).
unsigned long long wait_timeout_ns();

// Testing overrides set by gemm_testing_set_overrides (0 = not set): the
// CTA group of the BF16 launchers, and the clusters sharing a stream-K tail.
int testing_cta_group();
int testing_streamk_clusters();

// Encodes a rank-3 tiled TMA descriptor for a dense row-major tensor
// [d2][d1][d0] of `elem_bytes`-byte elements starting at `base`, with box
// {b0, b1, 1}, the given swizzle, zero fill for out-of-bounds elements.
// Returns GEMM_OK or GEMM_ERR_LAUNCH.
int encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* base,
                   uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1,
                   CUtensorMapSwizzle swizzle);

// Same, with explicit byte strides of dimensions 1 and 2 and a full 3-D box.
int encode_tmap_3d_strided(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                           uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                           uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2,
                           CUtensorMapSwizzle swizzle);

// Raster group height for the tile scheduler: consecutive work items walk
// `group_m` M blocks down one N column before moving right, so the A rows of
// a group are re-read from L2 across the N sweep and every B column block
// is fetched once per group.  As many M blocks as keep the group's A rows
// within 48 MB of the 129 MB L2 (all of them when A is small), at least 8.
inline int raster_group_m(int num_m_blocks, long long a_bytes_per_m_block) {
  const long long budget = 48ll << 20;
  long long g = a_bytes_per_m_block > 0 ? budget / a_bytes_per_m_block : num_m_blocks;
  if (g < 8) g = 8;
  if (g > num_m_blocks) g = num_m_blocks;
  return int(g < 1 ? 1 : g);
}

// Launchers; arguments are validated by the caller.
int launch_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, float scale,
                     bool scaled_acc, const DeviceInfo& dev, cudaStream_t stream);
// NN layout: B [K][N] row-major.
int launch_gemm_bf16_nn(const void* A, const void* B, void* C, int M, int N, int K,
                        const DeviceInfo& dev, cudaStream_t stream);
int launch_gemm_nvfp4(const void* a, const void* b, const void* sfa, const void* sfb, void* c,
                      int L, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream);
int launch_gemm_router(const void* A, const void* B, float* C, int M, int N, int K,
                       const DeviceInfo& dev, cudaStream_t stream);
int launch_scaled_add(void* out, const void* d, float scale, long n, const DeviceInfo& dev,
                      cudaStream_t stream);
int launch_selftest_timeout(int timeout_ms, const DeviceInfo& dev, cudaStream_t stream);

// Split-K: clamps `splits` to the number of 64-deep K blocks and returns the
// number of non-empty splits actually used (and the K blocks per split).
int splitk_effective_splits(int K, int splits, int* kb_per_split);
int launch_gemm_bf16_splitk(const void* A, const void* B, void* C, float* ws, int M, int N, int K,
                            int splits, const DeviceInfo& dev, cudaStream_t stream);
// NVFP4 split-K: S = min(k_splits, K/256) chunks of whole 256-deep K
// blocks, reduced so every chunk is non-empty; FP32 partials in
// ws[S][L][M][N], then an ordered reduce to FP16.
int nvfp4_splitk_effective_splits(int K, int splits, int* kb_per_split);
int launch_gemm_nvfp4_splitk(const void* a, const void* b, const void* sfa, const void* sfb,
                             void* c, float* ws, int L, int M, int N, int K, int splits,
                             const DeviceInfo& dev, cudaStream_t stream);
// Stream-K (CTA pairs, 256 x 256 tiles): at most streamk_max_clusters(dev)
// clusters, each with two FP32 partial tiles of workspace.
size_t streamk_max_clusters(const DeviceInfo& dev);
size_t streamk_workspace_bytes(const DeviceInfo& dev);
int launch_gemm_bf16_streamk(const void* A, const void* B, void* C, float* ws, int M, int N, int K,
                             const DeviceInfo& dev, cudaStream_t stream);
// W4A16: C = bf16(scale2 * (A . w^T)), w[n,k] = e2m1(b[n,k]) * e4m3(sfb[n,k/16]);
// b [N][K/2] (low nibble = even k), sfb [N][K/16]; K % 256 == 0, N % 8 == 0.
int launch_gemm_w4a16(const void* A, const uint8_t* b, const uint8_t* sfb, float scale2, void* C,
                      int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream);
// W4A16 with the transposed weight layout: b_t [K/2][ldb], sfb_t [K/16][ldb];
// K % 128 == 0, ldb % 16 == 0, ldb >= N, any N >= 1.
int launch_gemm_w4a16_t(const void* A, const uint8_t* b_t, const uint8_t* sfb_t, float scale2,
                        void* C, int M, int N, int K, int ldb, const DeviceInfo& dev,
                        cudaStream_t stream);
// Two-pass W4A16: weights converted into ws ([N][K] BF16), then the pair GEMM
// with the scale2 epilogue (launch_gemm_bf16_scale).
int launch_gemm_w4a16_twopass(const void* A, const uint8_t* b, const uint8_t* sfb, float scale2,
                              void* C, uint16_t* ws, int M, int N, int K, const DeviceInfo& dev,
                              cudaStream_t stream);
int launch_gemm_bf16_scale(const void* A, const void* B, void* C, int M, int N, int K,
                           float scale, const DeviceInfo& dev, cudaStream_t stream);
// C[i] = bf16(sum_{s=0..S-1} ws[s*n + i]) in split order (_f16: FP16).
int launch_splitk_reduce(const float* ws, void* C, size_t n, int splits, const DeviceInfo& dev,
                         cudaStream_t stream);
int launch_splitk_reduce_f16(const float* ws, void* C, size_t n, int splits, const DeviceInfo& dev,
                             cudaStream_t stream);

}  // namespace gb300
