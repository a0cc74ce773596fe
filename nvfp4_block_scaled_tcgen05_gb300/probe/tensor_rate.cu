// Tensor-pipe issue-rate probe (a measurement tool, not part of the GEMM
// library): how many SM cycles one CTA-pair tcgen05.mma takes when issued
// back to back, for the two MMA kinds the library uses, optionally with
// tcgen05.cp scale copies issued at the same time by other warps.
//
//   kind 0: tcgen05.mma.cta_group::2.kind::f16 (BF16), 256 x 256 x 16
//   kind 1: tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X,
//           256 x 256 x 64
//
// Each CTA pair zeroes 64 KB of shared memory (the operands: every MMA reads
// the same zero tiles, so only the issue and execution rate is measured, not
// the memory system), allocates 512 TMEM columns, and lane 0 of the leader's
// warp 1 issues `n_mma` MMAs into one accumulator, commits, and waits for
// them (bounded by %globaltimer).  With `copies` > 0, warps 2 and 3 of the
// leader together issue `copies` tcgen05.cp.32x128b.warpx4 per 4 MMAs into
// TMEM columns the MMAs do not use, from zeroed shared memory.
// out[2 * cluster] = SM cycles from the first MMA issue to the commit's
// completion (clock64 of the issuing SM), out[2 * cluster + 1] = the same
// interval in %globaltimer nanoseconds.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

namespace {

using namespace gb300;

constexpr int kSmemOperands = 64 * 1024;
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer() - t0 > kWaitNs) return false;
  return true;
}

__global__ void __launch_bounds__(128, 1)
    tensor_rate_kernel(int kind, int n_mma, int copies, unsigned long long* out,
                       unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  // barriers: MMAs done, and the copies of warp 2 and of warp 3 done; every
  // commit signals the leader CTA only (mask 1), which waits on all three
  const uint32_t bar_mma = sbase + kSmemOperands;
  auto bar_cp = [&](int w) { return bar_mma + 8u * uint32_t(w - 1); };  // warps 2, 3
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kSmemOperands + 32);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  for (int i = threadIdx.x; i < kSmemOperands / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_mma, 1);
    ptx::mbar_init(bar_cp(2), 1);
    ptx::mbar_init(bar_cp(3), 1);
    ptx::fence_mbar_init();
  }
  ptx::fence_proxy_async_smem();  // the zeroed operands, for the tensor core
  if (warp == 0) {
    ptx::tmem_alloc<2>(ptx::smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
    ptx::tmem_relinquish<2>();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // columns: accumulator 0..255, MMA scales 256..271, copy target 384..387
  const uint32_t sfa = tmem + 256, sfb = tmem + 264, cp_dst = tmem + 384;
  const uint64_t zero_desc = ptx::smem_desc(sbase + 32768, 0, 128, 0);  // 512 zero bytes
  if (rank == 0 && warp == 1 && lane == 0) {
    // zero scales (the block-scaled MMA reads them), then the timed MMAs
    if (kind == 1) {
      ptx::tc_cp_32x128b_warpx4<2>(sfa, zero_desc);
      ptx::tc_cp_32x128b_warpx4<2>(sfb, zero_desc);
      ptx::tc_cp_32x128b_warpx4<2>(sfb + 4, zero_desc);
    }
    const uint64_t adesc = ptx::sw128_kmajor_desc(sbase);
    const uint64_t bdesc = ptx::sw128_kmajor_desc(sbase + 16384);
    const uint32_t idesc = (kind == 1)
                               ? ((1u << 7) | (1u << 10) | (uint32_t(256 >> 3) << 17) |
                                  (uint32_t(256 >> 4) << 24))
                               : ((1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(256 >> 3) << 17) |
                                  (uint32_t(256 >> 4) << 24));
    const uint64_t g0 = ptx::globaltimer();
    const long long c0 = clock64();
    for (int i = 0; i < n_mma; ++i) {
      if (kind == 1) ptx::mma_nvf4<2>(tmem, adesc, bdesc, idesc, sfa, sfb, i > 0);
      else ptx::mma_bf16<2>(tmem, adesc, bdesc, idesc, i > 0);
    }
    ptx::tc_commit<2>(bar_mma, 1);
    const bool ok = wait_bounded(bar_mma, 0);
    const long long c1 = clock64();
    const uint64_t g1 = ptx::globaltimer();
    const int cluster = blockIdx.x / 2;
    out[2 * cluster] = ok ? (unsigned long long)(c1 - c0) : 0ull;
    out[2 * cluster + 1] = ok ? (g1 - g0) : 0ull;
    if (!ok) atomicCAS(status, 0u, 0x1A0u);
  } else if (rank == 0 && (warp == 2 || warp == 3) && lane == 0 && copies > 0) {
    const int n_cp = (n_mma / 4) * copies / 2;  // this warp's share
    for (int i = 0; i < n_cp; ++i) ptx::tc_cp_32x128b_warpx4<2>(cp_dst, zero_desc);
    ptx::tc_commit<2>(bar_cp(warp), 1);
    if (!wait_bounded(bar_cp(warp), 0)) atomicCAS(status, 0u, 0x1A1u);
  }
  // every tcgen05 operation is complete (each issuer waited for its commit)
  // before TMEM is freed
  ptx::tc_fence_before();
  ptx::cluster_sync();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<2>(tmem, 512);
  }
}

}  // namespace

// Returns 0 on success, 1 for bad arguments, 2 for a CUDA error, 3 when a
// bounded wait ran out.  `out` is a device buffer of 2 * clusters u64.
extern "C" __attribute__((visibility("default"))) int probe_tensor_rate(
    int kind, int clusters, int n_mma, int copies, unsigned long long* out, void* stream) {
  if (kind < 0 || kind > 1 || clusters < 1 || clusters > 1024 || n_mma < 4 || n_mma % 4 ||
      copies < 0 || copies > 64 || copies % 2 || !out)
    return 1;
  static unsigned int* status = nullptr;
  if (!status && cudaMalloc(&status, sizeof(unsigned int)) != cudaSuccess) return 2;
  if (cudaMemsetAsync(status, 0, sizeof(unsigned int), static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return 2;
  // more shared memory than two CTAs could share: one CTA (and one TMEM
  // allocation) per SM
  const int smem = 120 * 1024;
  if (cudaFuncSetAttribute(tensor_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return 2;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tensor_rate_kernel, kind, n_mma, copies, out, status) !=
      cudaSuccess)
    return 2;
  unsigned int st = 0;
  if (cudaMemcpyAsync(&st, status, sizeof st, cudaMemcpyDeviceToHost,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return 2;
  return st ? 3 : 0;
}
