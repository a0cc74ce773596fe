// Host-side launch of tcgen05_gemm_kernel instantiations: one-time per-device
// attributes, co-resident cluster count, cudaLaunchKernelEx with the cluster
// dimension of the configuration (its CTA group).
#pragma once

#include <algorithm>
#include <atomic>

#include "internal.h"
#include "tcgen05_gemm.cuh"

namespace gb300 {

// Testing overrides (gemm_testing_set_overrides): 0 lets the shape decide.
inline int cta_group_override() { return testing_cta_group(); }
inline int streamk_clusters_override() { return testing_streamk_clusters(); }

template <class Cfg, Epilogue EPI>
void fill_launch_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = Cfg::CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

// Clusters of this configuration that are co-resident on the device (at
// most one per SM group); sets the kernel's shared-memory attribute on first
// use.  Returns 0 when the attribute cannot be set.
template <class Cfg, Epilogue EPI>
int tcgen05_cluster_capacity(const DeviceInfo& dev) {
  static std::atomic<int> max_clusters[64];  // 0: not yet configured
  const int d = dev.device & 63;
  int cap = max_clusters[d].load();
  if (cap != 0) return cap;
  auto kern = tcgen05_gemm_kernel<Cfg, EPI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  fill_launch_config<Cfg, EPI>(cfg, attr, nullptr);
  cfg.gridDim = dim3(Cfg::CLUSTER * (dev.num_sms / Cfg::CLUSTER));
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = dev.num_sms / Cfg::CLUSTER;
  }
  cap = std::min(n, dev.num_sms / Cfg::CLUSTER);
  max_clusters[d].store(cap);
  return cap;
}

// Persistent launch: one cluster per co-resident slot, fewer when there are
// fewer tiles.  A stream-K schedule (p.sk) divides its tail over exactly
// `clusters` clusters, so the caller passes the count it planned with.
template <class Cfg, Epilogue EPI>
int launch_tcgen05(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                   const CUtensorMap& tsfa, const CUtensorMap& tsfb, const GemmParams& p,
                   const DeviceInfo& dev, cudaStream_t stream, int clusters = 0) {
  const int cap = tcgen05_cluster_capacity<Cfg, EPI>(dev);
  if (cap <= 0) return GEMM_ERR_LAUNCH;
  if (clusters <= 0) clusters = std::min(p.total_tiles, cap);
  if (clusters > cap) return GEMM_ERR_LAUNCH;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  fill_launch_config<Cfg, EPI>(cfg, attr, stream);
  // Programmatic dependent launch: the kernel's prologue (barrier set-up,
  // TMEM allocation, tensor-map prefetch) may overlap the end of the
  // previous kernel on the stream; every thread waits for that kernel's
  // completion before touching global memory.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(clusters * Cfg::CLUSTER);
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, tcgen05_gemm_kernel<Cfg, EPI>, ta, tb, tc, tsfa, tsfb, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // namespace gb300
