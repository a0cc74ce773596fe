// Tensor-pipe issue-rate probe (a measurement tool, not part of the GEMM
// library): how many SM cycles one CTA-pair tcgen05.mma takes when issued
// back to back, for the two MMA kinds the library uses, optionally with
// tcgen05.cp scale copies issued at the same time by other warps.
//
//   kind 0: tcgen05.mma.cta_group::2.kind::f16 (BF16), 256 x N x 16
//   kind 1: tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X,
//           256 x N x 64
// with N = 256 (the square tiles), 192 (the narrower BF16 tiles of
// under-filled shapes) or 128 (the decode tiles, whose N is the activation
// rows).
//
// Each CTA pair zeroes 64 KB of shared memory (the operands: every MMA reads
// the same zero tiles, so only the issue and execution rate is measured, not
// the memory system), allocates 512 TMEM columns, and lane 0 of the leader's
// warp 1 issues `n_mma` MMAs into one accumulator, commits, and waits for
// them (bounded by %globaltimer).  Warps 2 and 3 of the leader together
// issue, per 4 MMAs, `copies` tcgen05.cp.32x128b.warpx4 and `wide`
// tcgen05.cp.128x256b (half of each per warp) into TMEM columns the MMAs do
// not use, from zeroed shared memory.  With `commit_every` > 0 the issuers
// also commit as the GEMM kernel does per stage: the MMA thread after every
// `commit_every` MMAs, each copy warp after every group of copies (to the
// leader); every barrier of those commits expects all of them, and is
// waited for before the CTAs exit.  `flags` place waiting threads beside
// the MMAs, as the GEMM kernel's other roles are:
//   1: the MMA thread's intermediate commits go to both CTAs (multicast);
//      the peer CTA waits for them (as with 2)
//   2: the final commit goes to both CTAs and one thread of the peer CTA
//      waits for it from the start (it polls all through the MMAs)
//   4: the peer's waits sleep 256 ns between polls
//   8: one thread of the leader's warp 0 also waits for the final commit
//  16: with 8, all 32 lanes of that warp wait (as an epilogue warp does)
//  32: the leader's waiting warp sleeps 256 ns between polls
//  64: the commits follow a fixed pattern instead of a counter test:
//      groups of 4 MMAs (unrolled), the MMA thread commits after each
//      group (commit_every = 4)
// 128: as 64, but group g's commit is issued after the first MMA of group
//      g + 1 (the GEMM kernel's deferred stage release)
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

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, bool sleep = false) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > kWaitNs) return false;
    if (sleep) __nanosleep(256);
  }
  return true;
}

__global__ void __launch_bounds__(128, 1)
    tensor_rate_kernel(int kind, int mma_n, int n_mma, int copies, int wide, int commit_every,
                       int flags, unsigned long long* out, unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  // barriers: MMAs done, and the copies of warp 2 and of warp 3 done; every
  // commit signals the leader CTA only (mask 1), which waits on all three
  const uint32_t bar_mma = sbase + kSmemOperands;
  auto bar_cp = [&](int w) { return bar_mma + 8u * uint32_t(w - 1); };  // warps 2, 3
  // barriers of the intermediate commits: the MMA thread's (on both CTAs),
  // each copy warp's (on the leader)
  const uint32_t bar_mid = bar_mma + 40;
  auto bar_cpmid = [&](int w) { return bar_mma + 48u + 8u * uint32_t(w - 2); };
  const int n_groups = n_mma / 4;
  const bool grouped = (flags & (64 | 128)) != 0;
  const int n_mid = grouped ? n_mma / 4 - 1 : commit_every > 0 ? (n_mma - 1) / commit_every : 0;
  const int n_cpmid = (commit_every > 0 && copies + wide > 0) ? n_groups - 1 : 0;
  const bool mid_mcast = (flags & 1) != 0;
  const bool peer_waits = (flags & 2) || (mid_mcast && n_mid > 0);
  const bool peer_sleeps = (flags & 4) != 0;
  const bool leader_warp0_waits = (flags & 8) != 0;
  const bool leader_warp0_all = (flags & 16) != 0;
  const bool leader_sleeps = (flags & 32) != 0;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kSmemOperands + 32);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  for (int i = threadIdx.x; i < kSmemOperands / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_mma, 1);
    ptx::mbar_init(bar_cp(2), 1);
    ptx::mbar_init(bar_cp(3), 1);
    ptx::mbar_init(bar_mid, n_mid > 0 ? n_mid : 1);
    ptx::mbar_init(bar_cpmid(2), n_cpmid > 0 ? n_cpmid : 1);
    ptx::mbar_init(bar_cpmid(3), n_cpmid > 0 ? n_cpmid : 1);
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
  // columns: accumulator 0..255, MMA scales 256..271, copy targets 384..391
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
                               ? ((1u << 7) | (1u << 10) | (uint32_t(mma_n >> 3) << 17) |
                                  (uint32_t(256 >> 4) << 24))
                               : ((1u << 4) | (1u << 7) | (1u << 10) |
                                  (uint32_t(mma_n >> 3) << 17) | (uint32_t(256 >> 4) << 24));
    const uint64_t g0 = ptx::globaltimer();
    const long long c0 = clock64();
    auto mma = [&](uint32_t acc) {
      if (kind == 1) ptx::mma_nvf4<2>(tmem, adesc, bdesc, idesc, sfa, sfb, acc);
      else ptx::mma_bf16<2>(tmem, adesc, bdesc, idesc, acc);
    };
    const uint16_t mid_mask = mid_mcast ? 3 : 1;
    if (flags & 64) {
      for (int g = 0; g < n_mma / 4; ++g) {
#pragma unroll
        for (int j = 0; j < 4; ++j) mma(g > 0 || j > 0);
        if (g + 1 < n_mma / 4) ptx::tc_commit<2>(bar_mid, mid_mask);
      }
    } else if (flags & 128) {
      for (int g = 0; g < n_mma / 4; ++g) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          mma(g > 0 || j > 0);
          if (j == 0 && g > 0) ptx::tc_commit<2>(bar_mid, mid_mask);
        }
      }
    } else {
      for (int i = 0; i < n_mma; ++i) {
        mma(i > 0);
        if (commit_every > 0 && (i + 1) % commit_every == 0 && i + 1 < n_mma)
          ptx::tc_commit<2>(bar_mid, mid_mask);
      }
    }
    ptx::tc_commit<2>(bar_mma, peer_waits ? 3 : 1);
    bool ok = wait_bounded(bar_mma, 0);
    const long long c1 = clock64();
    const uint64_t g1 = ptx::globaltimer();
    const int cluster = blockIdx.x / 2;
    out[2 * cluster] = ok ? (unsigned long long)(c1 - c0) : 0ull;
    out[2 * cluster + 1] = ok ? (g1 - g0) : 0ull;
    if (!ok) atomicCAS(status, 0u, 0x1A0u);
    if (n_mid > 0 && !wait_bounded(bar_mid, 0)) atomicCAS(status, 0u, 0x1A2u);
  } else if (rank == 1 && warp == 1 && lane == 0 && peer_waits) {
    // the multicast commits also arrive here: all of them before exit
    if (!wait_bounded(bar_mma, 0, peer_sleeps)) atomicCAS(status, 0u, 0x1A0u);
    if (mid_mcast && n_mid > 0 && !wait_bounded(bar_mid, 0, peer_sleeps))
      atomicCAS(status, 0u, 0x1A2u);
  } else if (rank == 0 && warp == 0 && leader_warp0_waits && (lane == 0 || leader_warp0_all)) {
    if (!wait_bounded(bar_mma, 0, leader_sleeps)) atomicCAS(status, 0u, 0x1A4u);
  } else if (rank == 0 && (warp == 2 || warp == 3) && lane == 0 && copies + wide > 0) {
    // this warp's share: per 4 MMAs, copies / 2 narrow and wide / 2 wide ones
    for (int g = 0; g < n_groups; ++g) {
      for (int i = 0; i < copies / 2; ++i) ptx::tc_cp_32x128b_warpx4<2>(cp_dst, zero_desc);
      for (int i = 0; i < wide / 2; ++i) ptx::tc_cp_128x256b<2>(cp_dst, zero_desc);
      if (n_cpmid > 0 && g + 1 < n_groups) ptx::tc_commit<2>(bar_cpmid(warp), 1);
    }
    ptx::tc_commit<2>(bar_cp(warp), 1);
    if (!wait_bounded(bar_cp(warp), 0)) atomicCAS(status, 0u, 0x1A1u);
    if (n_cpmid > 0 && !wait_bounded(bar_cpmid(warp), 0)) atomicCAS(status, 0u, 0x1A3u);
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
    int kind, int mma_n, int clusters, int n_mma, int copies, int wide, int commit_every,
    int flags, unsigned long long* out, void* stream) {
  if (kind < 0 || kind > 1 || (mma_n != 128 && mma_n != 192 && mma_n != 256) || clusters < 1 ||
      clusters > 1024 || n_mma < 4 || n_mma % 4 || copies < 0 || copies > 64 || copies % 2 ||
      wide < 0 || wide > 16 || wide % 2 || commit_every < 0 || commit_every > 8192 || flags < 0 || flags > 255 ||
      (flags & 64 && flags & 128) || !out)
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
  if (cudaLaunchKernelEx(&cfg, tensor_rate_kernel, kind, mma_n, n_mma, copies, wide,
                         commit_every, flags, out, status) !=
      cudaSuccess)
    return 2;
  unsigned int st = 0;
  if (cudaMemcpyAsync(&st, status, sizeof st, cudaMemcpyDeviceToHost,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return 2;
  return st ? 3 : 0;
}
