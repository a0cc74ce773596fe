// BF16 NT GEMM and the fused scaled-acc (LoRA expand+fold) epilogue on
// tcgen05 kind::f16.  Tile 128 x 256 x 64, 4-stage TMA ring, two TMEM
// accumulators so the epilogue of one tile overlaps the next tile's K loop.
#include <algorithm>
#include <atomic>

#include "internal.h"
#include "tcgen05_gemm.cuh"

namespace gb300 {

using Bf16Cfg = TileCfg<Operand::kBF16, 256, 4>;

template <class Cfg, Epilogue EPI>
static int launch_tcgen05(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                          const GemmParams& p, const DeviceInfo& dev, cudaStream_t stream) {
  auto kern = tcgen05_gemm_kernel<Cfg, EPI>;
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = 1ull << (dev.device & 63);
  if (!(configured.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
        cudaSuccess)
      return GEMM_ERR_LAUNCH;
    configured.fetch_or(bit);
  }
  const int grid = std::min(p.total_tiles, dev.num_sms);
  kern<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(ta, tb, tc, p);
  return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

int launch_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, float scale,
                     bool scaled_acc, const DeviceInfo& dev, cudaStream_t stream) {
  using Cfg = Bf16Cfg;
  CUtensorMap ta, tb, tc;
  int rc = encode_tmap_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, uint64_t(K), uint64_t(M), 1,
                          64, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, uint64_t(K), uint64_t(N), 1,
                        64, Cfg::BN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, uint64_t(N), uint64_t(M), 1,
                        64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != GEMM_OK) return rc;
  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.L = 1;
  p.num_m_blocks = (M + Cfg::BM - 1) / Cfg::BM;
  p.num_n_blocks = (N + Cfg::BN - 1) / Cfg::BN;
  p.num_k_blocks = (K + Cfg::BK - 1) / Cfg::BK;
  p.total_tiles = p.num_m_blocks * p.num_n_blocks;
  p.scale = scale;
  p.status = dev.status;
  p.timeout_ns = wait_timeout_ns();
  return scaled_acc ? launch_tcgen05<Cfg, Epilogue::kScaledAccBF16>(ta, tb, tc, p, dev, stream)
                    : launch_tcgen05<Cfg, Epilogue::kStoreBF16>(ta, tb, tc, p, dev, stream);
}

}  // namespace gb300
