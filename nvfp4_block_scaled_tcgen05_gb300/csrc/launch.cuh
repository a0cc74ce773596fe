// Host-side launch of tcgen05_gemm_kernel instantiations: one-time per-device
// attributes, co-resident cluster count, cudaLaunchKernelEx with the cluster
// dimension of the configuration (CTA group x pairs sharing A).
#pragma once

#include <algorithm>
#include <atomic>
#include <cstdlib>

#include "internal.h"
#include "tcgen05_gemm.cuh"

namespace gb300 {

// CTA-group override for tests and experiments: GB300GEMM_CTA_GROUP=1 or 2
// forces that path when the shape allows it; anything else lets the shape decide.
inline int cta_group_override() {
  const char* e = std::getenv("GB300GEMM_CTA_GROUP");
  if (!e) return 0;
  const int v = std::atoi(e);
  return (v == 1 || v == 2) ? v : 0;
}

template <class Cfg, Epilogue EPI>
int launch_tcgen05(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                   const CUtensorMap& tsfa, const CUtensorMap& tsfb, const GemmParams& p,
                   const DeviceInfo& dev, cudaStream_t stream) {
  auto kern = tcgen05_gemm_kernel<Cfg, EPI>;
  static std::atomic<int> max_clusters[64];  // 0: not yet configured
  const int d = dev.device & 63;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = Cfg::CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters_cap = max_clusters[d].load();
  if (clusters_cap == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
        cudaSuccess)
      return GEMM_ERR_LAUNCH;
    int n = 0;
    cfg.gridDim = dim3(Cfg::CLUSTER * (dev.num_sms / Cfg::CLUSTER));
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = dev.num_sms / Cfg::CLUSTER;
    }
    clusters_cap = std::min(n, dev.num_sms / Cfg::CLUSTER);
    max_clusters[d].store(clusters_cap);
  }
  const int clusters = std::min(p.total_tiles, clusters_cap);
  cfg.gridDim = dim3(clusters * Cfg::CLUSTER);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tsfa, tsfb, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

}  // namespace gb300
