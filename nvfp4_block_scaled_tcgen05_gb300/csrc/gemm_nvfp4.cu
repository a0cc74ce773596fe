// NVFP4 block-scaled GEMM on tcgen05 kind::mxf4nvf4 (scale_vec::4X): packed
// e2m1 operands, one e4m3 scale per 16 K elements in the hardware scale
// layout ("kernelbot nvfp4 gemm submission 123329", sections "NVIDIA Block
// layout" / "Layout semantics"), FP16 output.  Tile 128 x 256 x 256, 3-stage
// ring; each stage also carries the 4 consecutive 512-byte scale atoms of
// the A rows and of each 128-row half of the B rows, which tcgen05.cp moves
// into a per-stage TMEM slot before the 4 MMAs of the stage.
#include <algorithm>
#include <atomic>

#include "internal.h"
#include "tcgen05_gemm.cuh"

namespace gb300 {

using Nvfp4Cfg = TileCfg<Operand::kNVFP4, 256, 3>;

int launch_gemm_nvfp4(const void* a, const void* b, const void* sfa, const void* sfb, void* c,
                      int L, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  using Cfg = Nvfp4Cfg;
  CUtensorMap ta, tb, tc;
  const uint64_t kb = uint64_t(K) / 2;  // bytes per packed row
  int rc = encode_tmap_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a, kb, uint64_t(M), uint64_t(L),
                          128, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b, kb, uint64_t(N), uint64_t(L), 128,
                        Cfg::BN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, c, uint64_t(N), uint64_t(M),
                        uint64_t(L), 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != GEMM_OK) return rc;
  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.L = L;
  p.num_m_blocks = M / Cfg::BM;
  p.num_n_blocks = (N + Cfg::BN - 1) / Cfg::BN;
  p.num_k_blocks = K / Cfg::BK;
  p.total_tiles = p.num_m_blocks * p.num_n_blocks * L;
  p.rest_m = M / 128;
  p.rest_n = N / 128;
  p.rest_k = K / 64;
  p.sfa = static_cast<const uint8_t*>(sfa);
  p.sfb = static_cast<const uint8_t*>(sfb);
  p.status = dev.status;
  p.timeout_ns = wait_timeout_ns();

  auto kern = tcgen05_gemm_kernel<Cfg, Epilogue::kStoreFP16>;
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

}  // namespace gb300
