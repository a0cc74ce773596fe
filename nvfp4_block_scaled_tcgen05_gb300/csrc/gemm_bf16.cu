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
// pipeline stages for output buffers (two halves per epilogue warp) so the
// old output of the next tile streams in while the current tile is written.
// The MMA sequence of a tile does not depend on the stage count, so every
// configuration with the same CTA group produces the same accumulators.
#include "launch.cuh"
#include "streamk.cuh"

namespace gb300 {

using Bf16Pair = TileCfg<Operand::kBF16, 2, 256, 6, 4, 2>;
using Bf16Single = TileCfg<Operand::kBF16, 1, 256, 4, 4, 2>;
// plain BF16 output: 128-deep stages (8 MMAs per stage), 3 stages
using Bf16PairStore = TileCfg<Operand::kBF16, 2, 256, 3, 4, 2, true, false, 2>;
// the same with 192-column tiles, for shapes whose 256-column tiles leave
// much of the last round of CTA pairs idle (see pair_tile_n)
using Bf16PairStore192 = TileCfg<Operand::kBF16, 2, 192, 3, 4, 2, true, false, 2>;
// NN layout (B stored [K][N]): the same tiles with B staged MN-major
using Bf16PairStoreNN = TileCfg<Operand::kBF16, 2, 256, 3, 4, 2, true, false, 2, true>;
using Bf16SingleNN = TileCfg<Operand::kBF16, 1, 256, 4, 4, 2, true, false, 1, true>;
// scaled-acc with K <= 256 (the LoRA fold): bound by streaming the output;
// 8 epilogue warps (each 128 of the 256 columns, 4 output buffers) keep more
// of that stream in flight than 4 (measured 75.9 -> 68.9 us at 4096 x 17408)
using Bf16PairStream = TileCfg<Operand::kBF16, 2, 256, 3, 8, 4>;
// K <= 64 (one K block per tile, e.g. LoRA rank 16): one operand stage is
// enough (a tile's single MMA takes ~160 cycles against microseconds of
// output streaming), and the freed 64 KB hold a third set of output boxes,
// so each warp requests the old output two tiles ahead
using Bf16PairStreamK1 = TileCfg<Operand::kBF16, 2, 256, 1, 8, 6>;
constexpr int kStreamK1MaxK = 64;
using Bf16SingleStream = TileCfg<Operand::kBF16, 1, 256, 2, 4, 8>;
constexpr int kStreamMaxK = 256;  // scaled-acc K up to this uses the streaming configurations

// Tensor maps and schedule of a BF16 launch writing C = A.B^T (or its
// scaled-acc update) tile by tile.
template <class Cfg>
static int setup_bf16(const void* A, const void* B, void* C, int M, int N, int K, float scale,
                      const DeviceInfo& dev, CUtensorMap& ta, CUtensorMap& tb, CUtensorMap& tc,
                      GemmParams& p) {
  int rc = encode_tmap_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, uint64_t(K), uint64_t(M), 1,
                          64, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
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
  p = GemmParams{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.L = 1;
  p.num_m_blocks = (M + Cfg::TILE_M - 1) / Cfg::TILE_M;
  p.num_n_blocks = (N + Cfg::BN - 1) / Cfg::BN;
  p.num_k_blocks = (K + Cfg::BK - 1) / Cfg::BK;
  p.total_tiles = p.num_m_blocks * p.num_n_blocks;
  p.group_m = raster_group_m(p.num_m_blocks, (long long)Cfg::TILE_M * K * 2);
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blocks;
  p.scale = scale;
  p.c_ptr = C;
  p.status = dev.status;
  p.timeout_ns = wait_timeout_ns();
  return GEMM_OK;
}

template <class Cfg>
static int run_bf16(const void* A, const void* B, void* C, int M, int N, int K, float scale,
                    bool scaled_acc, const DeviceInfo& dev, cudaStream_t stream) {
  CUtensorMap ta, tb, tc;
  GemmParams p;
  const int rc = setup_bf16<Cfg>(A, B, C, M, N, K, scale, dev, ta, tb, tc, p);
  if (rc != GEMM_OK) return rc;
  // the scale-factor maps are unused for BF16; pass A's map in their place
  if constexpr (Cfg::EPI_BUFS == 0) {
    return launch_tcgen05<Cfg, Epilogue::kStoreBF16>(ta, tb, tc, ta, ta, p, dev, stream);
  } else {
    return scaled_acc
               ? launch_tcgen05<Cfg, Epilogue::kScaledAccBF16>(ta, tb, tc, ta, ta, p, dev, stream)
               : launch_tcgen05<Cfg, Epilogue::kStoreBF16>(ta, tb, tc, ta, ta, p, dev, stream);
  }
}

// Clusters sharing the stream-K tail, or 0 for the data-parallel schedule.
// Dividing the tail pays when the last round leaves most clusters idle: with
// a quarter or more of them busy, GB300 runs the short round about as fast
// per tile as a full one (measured), and the partial tiles cost more than
// they save.  P then follows the cost model of streamk_min_cost_share.  A
// testing override (gemm_testing_set_overrides) forces the division over
// min(P, C) clusters.
static int streamk_share(int tiles, int kbt, int C) {
  if (const int v = streamk_clusters_override()) return v < C ? v : C;
  const int tail = tiles % C;
  if (tail == 0 || 4 * tail > C) return 0;
  return streamk_min_cost_share((long long)tail * kbt, tail, C);
}

// Stream-K over exactly the co-resident cluster count C: floor(tiles / C)
// data-parallel rounds of whole tiles, then the remaining tiles' K
// iterations split evenly over P <= C clusters (each writes at most two
// FP32 partial tiles to ws), then the ordered fixup of the split tiles.
template <class Cfg>
static int run_bf16_streamk(const void* A, const void* B, void* C, float* ws, int M, int N, int K,
                            const DeviceInfo& dev, cudaStream_t stream) {
  static_assert(!Cfg::kRegEpi && Cfg::EPI_BUFS > 0,
                "partial tiles are written by the TMA-store epilogue");
  CUtensorMap ta, tb, tc, tw;
  GemmParams p;
  int rc = setup_bf16<Cfg>(A, B, C, M, N, K, 0.0f, dev, ta, tb, tc, p);
  if (rc != GEMM_OK) return rc;
  const int clusters = tcgen05_cluster_capacity<Cfg, Epilogue::kStoreBF16>(dev);
  if (clusters <= 0) return GEMM_ERR_LAUNCH;
  if (size_t(clusters) > streamk_max_clusters(dev) || clusters > kSkMaxTail)
    return GEMM_ERR_LAUNCH;
  // workspace: [clusters * 2][TILE_M][BN] FP32, stored in 32 x 32 boxes
  rc = encode_tmap_3d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ws, uint64_t(Cfg::BN),
                      uint64_t(Cfg::TILE_M), uint64_t(clusters) * 2, 32, 32,
                      CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != GEMM_OK) return rc;
  p.sk = streamk_share(p.total_tiles, p.num_k_blocks, clusters);
  {
    // no cluster without tail work: P <= T
    const long long T = (long long)(p.total_tiles % clusters) * p.num_k_blocks;
    if (p.sk > T) p.sk = int(T);
  }
  rc = launch_tcgen05<Cfg, Epilogue::kStoreBF16>(ta, tb, tc, tw, ta, p, dev, stream,
                                                 p.sk ? clusters : 0);
  if (rc != GEMM_OK) return rc;
  if (p.sk == 0) return GEMM_OK;
  StreamKPlan plan;
  build_streamk_plan<Cfg>(p, clusters, plan);
  if (plan.tiles == 0) return GEMM_OK;
  return launch_streamk_fixup<Cfg>(plan, p, ws, stream);
}

size_t streamk_max_clusters(const DeviceInfo& dev) { return size_t(dev.num_sms / 2); }

size_t streamk_workspace_bytes(const DeviceInfo& dev) {
  return streamk_max_clusters(dev) * 2 * Bf16PairStore::TILE_M * Bf16PairStore::BN * sizeof(float);
}

int launch_gemm_bf16_streamk(const void* A, const void* B, void* C, float* ws, int M, int N, int K,
                             const DeviceInfo& dev, cudaStream_t stream) {
  return run_bf16_streamk<Bf16PairStore>(A, B, C, ws, M, N, K, dev, stream);
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

// C = bf16(scale * A.B^T) on the plain-output pair configuration (the
// epilogue of the W4A16 GEMM, whose tiles and K order it shares).
int launch_gemm_bf16_scale(const void* A, const void* B, void* C, int M, int N, int K,
                           float scale, const DeviceInfo& dev, cudaStream_t stream) {
  using Cfg = Bf16PairStore;
  CUtensorMap ta, tb, tc;
  GemmParams p;
  const int rc = setup_bf16<Cfg>(A, B, C, M, N, K, scale, dev, ta, tb, tc, p);
  if (rc != GEMM_OK) return rc;
  return launch_tcgen05<Cfg, Epilogue::kScaleBF16>(ta, tb, tc, ta, ta, p, dev, stream);
}

int launch_gemm_bf16_nn(const void* A, const void* B, void* C, int M, int N, int K,
                        const DeviceInfo& dev, cudaStream_t stream) {
  int cg = (M > 128) ? 2 : 1;
  if (const int o = cta_group_override()) cg = o;
  return cg == 2 ? run_bf16<Bf16PairStoreNN>(A, B, C, M, N, K, 0.0f, false, dev, stream)
                 : run_bf16<Bf16SingleNN>(A, B, C, M, N, K, 0.0f, false, dev, stream);
}

// Column width of the plain-output pair tiles: 256 or 192, whichever gives
// the shorter critical path = rounds of tiles over the CTA pairs x cycles of
// one pair MMA at that width (measured: 162.3 cycles for 256x256x16, 130.3
// for 256x192x16; bench.py --tensor-rate).  192-column tiles re-read A
// more, but on shapes whose 256-wide tiles fill the pairs badly they win:
// 5120x512x2048 16.3 -> 13.9 us (60 tiles instead of 40 on 76 pairs),
// 5120x2048x2048 34.7 -> 31.4 us and 5120x2048x11008 158.9 -> 142.9 us
// (220 tiles in 3 rounds instead of 160 in 3); gate/up (860 vs 1160
// tiles) stays at 256.  Results are the same at either width (the K loop
// of every output is the same).
static int pair_tile_n(int M, int N, const DeviceInfo& dev) {
  const long long pairs = dev.num_sms / 2;
  const long long mb = (M + 255) / 256;
  auto path = [&](int bn, double mma_cycles) {
    const long long tiles = mb * ((N + bn - 1) / bn);
    return double((tiles + pairs - 1) / pairs) * mma_cycles;
  };
  return path(192, 130.3) < path(256, 162.3) ? 192 : 256;
}

int launch_gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, float scale,
                     bool scaled_acc, const DeviceInfo& dev, cudaStream_t stream) {
  const long long pair_tiles = (long long)((M + 255) / 256) * ((N + 255) / 256);
  int cg = (pair_tiles >= dev.num_sms / 2) ? 2 : 1;
  if (const int o = cta_group_override()) cg = o;
  if (scaled_acc && K <= kStreamMaxK) {
    if (cg == 2 && K <= kStreamK1MaxK)
      return run_bf16<Bf16PairStreamK1>(A, B, C, M, N, K, scale, true, dev, stream);
    return cg == 2 ? run_bf16<Bf16PairStream>(A, B, C, M, N, K, scale, true, dev, stream)
                   : run_bf16<Bf16SingleStream>(A, B, C, M, N, K, scale, true, dev, stream);
  }
  // Plain outputs: a CTA pair covers 256 rows with the same per-SM work as
  // one CTA on 128 rows, so pairs (128-deep stages, half the B traffic per
  // SM) occupy as many SMs as single CTAs whenever M spans two row blocks.
  if (!scaled_acc && !cta_group_override()) cg = (M > 128) ? 2 : 1;
  if (!scaled_acc && cg == 2)
    return pair_tile_n(M, N, dev) == 192
               ? run_bf16<Bf16PairStore192>(A, B, C, M, N, K, 0.0f, false, dev, stream)
               : run_bf16<Bf16PairStore>(A, B, C, M, N, K, 0.0f, false, dev, stream);
  return cg == 2 ? run_bf16<Bf16Pair>(A, B, C, M, N, K, scale, scaled_acc, dev, stream)
                 : run_bf16<Bf16Single>(A, B, C, M, N, K, scale, scaled_acc, dev, stream);
}

}  // namespace gb300
