// BF16 NT GEMM and the fused scaled-acc (LoRA expand+fold) epilogue on
// tcgen05 kind::f16, FP32 accumulation in TMEM.
//
// Two tile configurations, chosen per shape:
//  * pair (cta_group::2): 256 x 256 tiles shared by two SMs, each staging its
//    128 A rows and 128 of the 256 B rows per 64-deep K step (32 KB per stage,
//    6 stages), two TMEM accumulators per CTA;
//  * single (cta_group::1): 128 x 256 tiles, 48 KB stages, 4 stages; used when
//    there are fewer pair tiles than SM pairs.
// The scaled-acc epilogue of a short-K GEMM (the LoRA fold, K = rank) is
// bound by reading and writing the output; its configurations trade
// pipeline stages for eight output buffers per epilogue warp so the old
// output of the next tile streams in while the current tile is written.
// The MMA sequence of a tile does not depend on the stage count, so every
// configuration with the same CTA group produces the same accumulators.
#include <cstdlib>

#include "launch.cuh"

namespace gb300 {

using Bf16Pair = TileCfg<Operand::kBF16, 2, 256, 6, 4, 2>;
using Bf16Single = TileCfg<Operand::kBF16, 1, 256, 4, 4, 2>;
// plain BF16 output: 128-deep stages (8 MMAs per stage), 3 stages
using Bf16PairStore = TileCfg<Operand::kBF16, 2, 256, 3, 4, 2, true, false, 1, 2>;
// NN layout (B stored [K][N]): the same tiles with B staged MN-major
using Bf16PairStoreNN = TileCfg<Operand::kBF16, 2, 256, 3, 4, 2, true, false, 1, 2, true>;
using Bf16SingleNN = TileCfg<Operand::kBF16, 1, 256, 4, 4, 2, true, false, 1, 1, true>;
// two pairs per cluster sharing (multicasting) their A rows
using Bf16PairMC = TileCfg<Operand::kBF16, 2, 256, 6, 4, 2, true, false, 2>;
using Bf16PairStream = TileCfg<Operand::kBF16, 2, 256, 3, 4, 8>;
using Bf16SingleStream = TileCfg<Operand::kBF16, 1, 256, 2, 4, 8>;
constexpr int kStreamMaxK = 256;  // scaled-acc K up to this uses the streaming configurations

template <class Cfg>
static int run_bf16(const void* A, const void* B, void* C, int M, int N, int K, float scale,
                    bool scaled_acc, const DeviceInfo& dev, cudaStream_t stream) {
  CUtensorMap ta, tb, tc;
  int rc = encode_tmap_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, uint64_t(K), uint64_t(M), 1,
                          64, Cfg::A_SLICE_ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == GEMM_OK) {
    if constexpr (Cfg::B_MN)  // B [K][N]: boxes of 64 columns x BK rows
      rc = encode_tmap_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, uint64_t(N), uint64_t(K), 1,
                          64, Cfg::BK, CU_TENSOR_MAP_SWIZZLE_128B);
    else
      rc = encode_tmap_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, uint64_t(K), uint64_t(N), 1,
                          64, Cfg::B_ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, uint64_t(N), uint64_t(M), 1,
                        64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != GEMM_OK) return rc;
  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.L = 1;
  p.num_m_blocks = (M + Cfg::TILE_M - 1) / Cfg::TILE_M;
  p.num_n_blocks = (N + Cfg::BN - 1) / Cfg::BN;
  p.num_k_blocks = (K + Cfg::BK - 1) / Cfg::BK;
  p.total_tiles = p.num_m_blocks * ((p.num_n_blocks + Cfg::MC - 1) / Cfg::MC);
  p.group_m = raster_group_m(p.num_m_blocks, (long long)Cfg::TILE_M * K * 2);
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blocks;
  p.scale = scale;
  p.c_ptr = C;
  p.status = dev.status;
  p.timeout_ns = wait_timeout_ns();
  // the scale-factor maps are unused for BF16; pass A's map in their place
  if constexpr (Cfg::EPI_BUFS == 0) {
    return launch_tcgen05<Cfg, Epilogue::kStoreBF16>(ta, tb, tc, ta, ta, p, dev, stream);
  } else {
    return scaled_acc
               ? launch_tcgen05<Cfg, Epilogue::kScaledAccBF16>(ta, tb, tc, ta, ta, p, dev, stream)
               : launch_tcgen05<Cfg, Epilogue::kStoreBF16>(ta, tb, tc, ta, ta, p, dev, stream);
  }
}

// Split-K: split s of the K blocks [s*kbps, (s+1)*kbps) writes its FP32
// partial tile into workspace[s][M][N]; a second kernel sums the splits in
// order s = 0..S-1 and rounds to BF16 ("gemm_dense.rs", dense_gemm_splitk).
template <class Cfg>
static int run_bf16_splitk(const void* A, const void* B, float* ws, int M, int N, int K,
                           int splits, int kbps, const DeviceInfo& dev, cudaStream_t stream) {
  CUtensorMap ta, tb, tw;
  int rc = encode_tmap_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, uint64_t(K), uint64_t(M), 1,
                          64, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, uint64_t(K), uint64_t(N), 1,
                        64, Cfg::B_ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, uint64_t(N), uint64_t(M),
                        uint64_t(splits), 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != GEMM_OK) return rc;
  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.L = splits;
  p.num_m_blocks = (M + Cfg::TILE_M - 1) / Cfg::TILE_M;
  p.num_n_blocks = (N + Cfg::BN - 1) / Cfg::BN;
  p.num_k_blocks = (K + Cfg::BK - 1) / Cfg::BK;
  p.total_tiles = p.num_m_blocks * p.num_n_blocks * splits;
  p.group_m = raster_group_m(p.num_m_blocks, (long long)Cfg::TILE_M * K * 2);
  p.k_splits = splits;
  p.kb_per_split = kbps;
  p.status = dev.status;
  p.timeout_ns = wait_timeout_ns();
  return launch_tcgen05<Cfg, Epilogue::kStoreF32>(ta, tb, tw, ta, ta, p, dev, stream);
}

int splitk_effective_splits(int K, int splits, int* kb_per_split) {
  const int nkb = (K + 63) / 64;
  if (splits > nkb) splits = nkb;
  const int kbps = (nkb + splits - 1) / splits;
  *kb_per_split = kbps;
  return (nkb + kbps - 1) / kbps;  // every split non-empty
}

int launch_gemm_bf16_splitk(const void* A, const void* B, void* C, float* ws, int M, int N, int K,
                            int splits, const DeviceInfo& dev, cudaStream_t stream) {
  int kbps = 0;
  const int s_eff = splitk_effective_splits(K, splits, &kbps);
  const long long pair_units = (long long)((M + 255) / 256) * ((N + 255) / 256) * s_eff;
  int cg = (pair_units >= dev.num_sms / 2) ? 2 : 1;
  if (const int o = cta_group_override()) cg = o;
  const int rc = cg == 2 ? run_bf16_splitk<Bf16Pair>(A, B, ws, M, N, K, s_eff, kbps, dev, stream)
                         : run_bf16_splitk<Bf16Single>(A, B, ws, M, N, K, s_eff, kbps, dev, stream);
  if (rc != GEMM_OK) return rc;
  return launch_splitk_reduce(ws, C, size_t(M) * N, s_eff, dev, stream);
}

int launch_gemm_bf16_nn(const void* A, const void* B, void* C, int M, int N, int K,
                        const DeviceInfo& dev, cudaStream_t stream) {
  int cg = (M > 128) ? 2 : 1;
  if (const int o = cta_group_override()) cg = o;
  return cg == 2 ? run_bf16<Bf16PairStoreNN>(A, B, C, M, N, K, 0.0f, false, dev, stream)
                 : run_bf16<Bf16SingleNN>(A, B, C, M, N, K, 0.0f, false, dev, stream);
}

int launch_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, float scale,
                     bool scaled_acc, const DeviceInfo& dev, cudaStream_t stream) {
  const long long pair_tiles = (long long)((M + 255) / 256) * ((N + 255) / 256);
  int cg = (pair_tiles >= dev.num_sms / 2) ? 2 : 1;
  if (const int o = cta_group_override()) cg = o;
  if (scaled_acc && K <= kStreamMaxK)
    return cg == 2 ? run_bf16<Bf16PairStream>(A, B, C, M, N, K, scale, true, dev, stream)
                   : run_bf16<Bf16SingleStream>(A, B, C, M, N, K, scale, true, dev, stream);
  // Plain outputs: a CTA pair covers 256 rows with the same per-SM work as
  // one CTA on 128 rows, so pairs (128-deep stages, half the B traffic per
  // SM) occupy as many SMs as single CTAs whenever M spans two row blocks.
  if (!scaled_acc && !cta_group_override()) cg = (M > 128) ? 2 : 1;
  if (!scaled_acc && cg == 2) {
    // GB300GEMM_MC=2 selects the A-multicast cluster; measured no faster
    // than the plain pair on the shapes here (GB300), so it is opt-in.
    const char* e = std::getenv("GB300GEMM_MC");
    const bool mc = e && std::atoi(e) == 2;
    if (mc && (N + 255) / 256 >= 2)
      return run_bf16<Bf16PairMC>(A, B, C, M, N, K, 0.0f, false, dev, stream);
    return run_bf16<Bf16PairStore>(A, B, C, M, N, K, 0.0f, false, dev, stream);
  }
  return cg == 2 ? run_bf16<Bf16Pair>(A, B, C, M, N, K, scale, scaled_acc, dev, stream)
                 : run_bf16<Bf16Single>(A, B, C, M, N, K, scale, scaled_acc, dev, stream);
}

}  // namespace gb300
