// NVFP4 block-scaled GEMM on tcgen05 kind::mxf4nvf4 (scale_vec::4X): packed
// e2m1 operands, one e4m3 scale per 16 K elements in the hardware scale
// layout ("kernelbot nvfp4 gemm submission 123329", sections "NVIDIA Block
// layout" / "Layout semantics"), FP16 output.
//
// Each 256-element K stage carries, per 128 rows, the 4 consecutive 512-byte
// scale atoms of that K range (2 KB, contiguous in the hardware layout),
// which tcgen05.cp moves into a per-stage TMEM slot before the stage's 4
// MMAs.  The MMA reads the scales of row 32*i + g from TMEM lane 32*i + g,
// column base + i, so an atom has to land in all four 32-lane quarters:
// the 32x128b.warpx4 copy replicates one atom into them (12 copies per
// stage for a 256-row B tile).  The FP32-partial and decode configurations
// instead stage the A atoms four times in shared memory (one TMA box whose
// replica dimension has stride 0), so that one 128-lane x 32-byte copy
// fills the scale columns of two MMAs.  Two dedicated warps share every
// stage's copies (MMAs 0-1 and 2-3) and both arrive on the stage's barrier,
// so the MMA thread issues only MMAs and a stage whose data lands just in
// time waits for half of the copies' issue time (each tcgen05 instruction
// costs the issuing thread about 60 cycles).
// One TMEM accumulator (256 columns) plus the scale slots fill the 512
// columns, so the epilogue is register-staged: 8 warps read the whole
// accumulator, release it, then convert it into per-warp boxes in shared
// memory that TMA writes out, while the next tile's MMAs run.
//
// Configuration: CTA pairs (cta_group::2, 256 x 256 tiles, each CTA stages
// its 128 A rows, 128 B rows and the scales of all 256 B rows, 5 stages)
// for every shape with M > 256; with M = 128 the second CTA's rows would lie
// past M, so decode-like problems swap the operands (below).  A single-CTA
// configuration (cta_group::1, 128 x 256 tiles, 3 stages, scale-copy warps)
// faulted the GPU twice when launched back to back; the cause was not
// found, so it is not used.
// Split-K (decode-like M = 128 with few output tiles): FP32 partials of
// K-block chunks go into a caller workspace, then an ordered reduce rounds
// once to FP16 ("gemm_dense.rs", dense_gemm_splitk, applied to the
// block-scaled GEMM).  With M <= 256 the operands swap roles (D = B . A^T,
// the weights on the 256-row MMA side of the CTA pair, the activation rows
// as MMA N = 128) and the epilogue writes D transposed, one 32 x 32 FP32
// box per warp by TMA: no MMA rows are spent on zero fill, and the
// 256-row weight tiles times the splits give enough work units for the
// CTA pairs.
#include "launch.cuh"

namespace gb300 {

// FP16 output: unreplicated A scales (6 KB less per stage), which leaves
// room to stage the output in shared memory and write it by TMA (direct
// 16-byte stores into 32 rows per warp instruction slowed the next tile's
// first stages by about 5000 cycles per tile)
using Nvfp4Pair = TileCfg<Operand::kNVFP4, 2, 256, 5, 8, 1, false, false>;
// FP32 split-K partials (M > 256): replicated A scales, partials stored
// straight from registers
using Nvfp4PairPartials = TileCfg<Operand::kNVFP4, 2, 256, 5, 8, 0, true, false>;
// Decode-like problems (M <= 256 activation rows): the operands swap roles,
// so the weights fill the 256-row MMA M side of a CTA pair and the
// activation rows are the MMA N = 128; the output is stored transposed.
using Nvfp4PairT = TileCfg<Operand::kNVFP4, 2, 128, 6, 4, 1, true, false, 1, false, true>;

// `out` is the FP16 output (EPI = kStoreFP16) or, with splits > 1 (L = 1),
// the FP32 workspace [splits][M][N] (EPI = kStoreF32).
template <class Cfg, Epilogue EPI = Epilogue::kStoreFP16>
static int run_nvfp4(const void* a, const void* b, const void* sfa, const void* sfb, void* out,
                     int L, int M, int N, int K, int splits, int kb_per_split,
                     const DeviceInfo& dev, cudaStream_t stream) {
  void* c = out;
  CUtensorMap ta, tb, tc, tsa, tsb;
  const uint64_t kb = uint64_t(K) / 2;  // bytes per packed row
  const int rest_m = M / 128, rest_n = N / 128, rest_k = K / 64;
  int rc = encode_tmap_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a, kb, uint64_t(M), uint64_t(L),
                          128, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b, kb, uint64_t(N), uint64_t(L), 128,
                        Cfg::B_ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == GEMM_OK) {
    if constexpr (Cfg::C_T) {
      // transposed output [slot][N][M] (M = the weights, innermost), 32 x 32
      // boxes; slot = batch, or split * L + batch for FP32 partials
      const bool f32 = (EPI == Epilogue::kStoreF32);
      rc = encode_tmap_3d(&tc, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          f32 ? 4 : 2, c, uint64_t(M), uint64_t(N),
                          uint64_t(splits > 1 ? splits * L : L), 32, 32,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
      rc = encode_tmap_3d(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, c, uint64_t(N), uint64_t(M),
                          uint64_t(L), 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    }
  }
  // scales: one row of rest_k * 512 bytes (= rest_k * 64 u64) per (l, 128-row block)
  if (rc == GEMM_OK) {
    if constexpr (Cfg::SFA_REP) {
      // [atom][replica][64 u64]: the replica dimension has stride 0, so one
      // box of 4 x 4 x 512 B stages each of a stage's 4 atoms four times.
      rc = encode_tmap_3d_strided(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT64, sfa, 64, 4,
                                  uint64_t(L) * rest_m * rest_k, 0, 512, 64, 4, 4,
                                  CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
      rc = encode_tmap_3d(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT64, 8, sfa, uint64_t(rest_k) * 64,
                          uint64_t(L) * rest_m, 1, 256, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
  }
  if (rc == GEMM_OK)
    rc = Cfg::SFB_REP
             ? encode_tmap_3d_strided(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT64, sfb, 64, 4,
                                      uint64_t(L) * rest_n * rest_k, 0, 512, 64, 4, 4,
                                      CU_TENSOR_MAP_SWIZZLE_NONE)
             : encode_tmap_3d(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT64, 8, sfb, uint64_t(rest_k) * 64,
                              uint64_t(L) * rest_n, 1, 256, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != GEMM_OK) return rc;
  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.L = splits > 1 ? splits * L : L;  // split-K: batch slot = batch * splits + split
  p.num_m_blocks = (M + Cfg::TILE_M - 1) / Cfg::TILE_M;
  p.num_n_blocks = (N + Cfg::BN - 1) / Cfg::BN;
  p.num_k_blocks = K / Cfg::BK;
  p.total_tiles = p.num_m_blocks * p.num_n_blocks * p.L;
  p.group_m = raster_group_m(p.num_m_blocks, (long long)Cfg::TILE_M * (K / 2 + K / 16));
  p.k_splits = splits;
  p.kb_per_split = splits > 1 ? kb_per_split : p.num_k_blocks;
  p.rest_m = rest_m;
  p.rest_n = rest_n;
  p.rest_k = rest_k;
  p.c_ptr = c;
  p.status = dev.status;
  p.timeout_ns = wait_timeout_ns();
  return launch_tcgen05<Cfg, EPI>(ta, tb, tc, tsa, tsb, p, dev, stream);
}

constexpr int kNvfp4SwapMaxM = 256;  // activation rows up to this use the swapped kernel

int launch_gemm_nvfp4(const void* a, const void* b, const void* sfa, const void* sfb, void* c,
                      int L, int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  return run_nvfp4<Nvfp4Pair>(a, b, sfa, sfb, c, L, M, N, K, 1, 0, dev, stream);
}

int nvfp4_splitk_effective_splits(int K, int splits, int* kb_per_split) {
  const int nkb = K / Nvfp4Pair::BK;
  if (splits > nkb) splits = nkb;
  const int kbps = (nkb + splits - 1) / splits;
  *kb_per_split = kbps;
  return (nkb + kbps - 1) / kbps;  // every split non-empty
}

int launch_gemm_nvfp4_splitk(const void* a, const void* b, const void* sfa, const void* sfb,
                             void* c, float* ws, int L, int M, int N, int K, int splits,
                             const DeviceInfo& dev, cudaStream_t stream) {
  int kbps = 0;
  const int s_eff = nvfp4_splitk_effective_splits(K, splits, &kbps);
  // partials ws[split][batch][M][N] in FP32, either orientation
  const int rc =
      (M <= kNvfp4SwapMaxM)
          ? run_nvfp4<Nvfp4PairT, Epilogue::kStoreF32>(b, a, sfb, sfa, ws, L, N, M, K, s_eff, kbps,
                                                        dev, stream)
          : run_nvfp4<Nvfp4PairPartials, Epilogue::kStoreF32>(a, b, sfa, sfb, ws, L, M, N, K,
                                                               s_eff, kbps, dev, stream);
  if (rc != GEMM_OK) return rc;
  return launch_splitk_reduce_f16(ws, c, size_t(L) * M * N, s_eff, dev, stream);
}

}  // namespace gb300
