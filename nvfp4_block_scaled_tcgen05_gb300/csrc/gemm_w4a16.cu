// W4A16 GEMM: C[M,N] = bf16( scale2 * A[M,K] . w^T ), w = e2m1 * e4m3 the
// NVFP4 weights of "gemm_dense.rs" w4a16_gemm (e2m1 codes, e4m3 block
// scales, an FP32 per-tensor scale), on the persistent tcgen05 kernel: CTA
// pairs, 256 x 256 tiles, 3 stages of 128 K values.  A is staged by TMA into
// the stages; the packed codes and block scales by TMA into a 3-deep ring of
// their own; eight warps per CTA turn the pair's 256 weight rows of each
// stage into exact BF16 in the stage; the MMAs are the BF16 kind::f16 MMAs of the
// dense GEMM; the epilogue multiplies the FP32 sum by scale2 once.  The
// weights are read once per tile from L2/HBM at 4.5 bits each instead of 16.
#include <algorithm>

#include "launch.cuh"

namespace gb300 {

// One 16-row output box per epilogue warp (8 KB) beside the stages and a
// 2-deep code / scale ring: the output goes out by TMA.  Direct 16-byte
// stores from registers measured 54.2 us at 1016 x 12288 x 2048 against
// 46.4 us with no output stores at all; a 2-deep ring measured the same
// as a 3-deep one (54.2 us).
using W4Pair = TileCfg<Operand::kW4A16, 2, 256, 3, 4, 1, true, false, 2>;
// the transposed weight layout: the same tiles and MMA sequence with B
// staged MN-major (as the NN GEMM stages it); any N, so rows of C that are
// not 16-byte aligned (N % 8 != 0) take the direct-store epilogue
using W4PairT = TileCfg<Operand::kW4A16, 2, 256, 3, 4, 1, true, false, 2, true>;
using W4PairTDirect = TileCfg<Operand::kW4A16, 2, 256, 3, 4, 0, true, false, 2, true>;

int launch_gemm_w4a16(const void* A, const uint8_t* b, const uint8_t* sfb, float scale2, void* C,
                      int M, int N, int K, const DeviceInfo& dev, cudaStream_t stream) {
  using Cfg = W4Pair;
  CUtensorMap ta, tcode, tscale, tc;
  int rc = encode_tmap_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, uint64_t(K), uint64_t(M), 1,
                          64, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
  // codes: N rows of K/2 bytes, 64-byte x B_ROWS boxes (one K block of the
  // CTA's weight rows); scales: N rows of K/16 bytes, 16-byte boxes
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tcode, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b, uint64_t(K / 2), uint64_t(N),
                        1, 64, Cfg::B_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tscale, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, sfb, uint64_t(K / 16),
                        uint64_t(N), 1, 16, Cfg::B_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, uint64_t(N), uint64_t(M), 1,
                        64, Cfg::EPI_BOX_ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != GEMM_OK) return rc;
  GemmParams p{};
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
  p.scale = scale2;
  p.c_ptr = C;
  p.status = dev.status;
  p.timeout_ns = wait_timeout_ns();
  // the A-scale map is unused; pass A's map in its place
  return launch_tcgen05<Cfg, Epilogue::kScaleBF16>(ta, tcode, tc, ta, tscale, p, dev, stream);
}

// Transposed weight layout ("gemm_dense.rs", w4a16_gemm_n128_ldb and
// w4a16_gemm_n128_m128_bf16): codes b_t [K/2][ldb] bytes (byte (j, n) =
// elements 2j, 2j+1 of column n), scales sfb_t [K/16][ldb]; ldb % 16 == 0,
// K % 128 == 0, any N >= 1 (C rows are then 2N bytes apart).
template <class Cfg>
static int run_w4a16_t(const void* A, const uint8_t* b_t, const uint8_t* sfb_t, float scale2,
                       void* C, int M, int N, int K, int ldb, const DeviceInfo& dev,
                       cudaStream_t stream) {
  CUtensorMap ta, tcode, tscale, tc;
  int rc = encode_tmap_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, uint64_t(K), uint64_t(M), 1,
                          64, Cfg::BM, CU_TENSOR_MAP_SWIZZLE_128B);
  // codes: K/2 rows of ldb bytes, boxes of B_ROWS columns x 64 rows (one
  // 128-deep K block of the CTA's columns); scales: K/16 rows, 8-row boxes
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tcode, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b_t, uint64_t(ldb),
                        uint64_t(K / 2), 1, Cfg::B_ROWS, 64, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc == GEMM_OK)
    rc = encode_tmap_3d(&tscale, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, sfb_t, uint64_t(ldb),
                        uint64_t(K / 16), 1, Cfg::B_ROWS, 8, CU_TENSOR_MAP_SWIZZLE_NONE);
  if constexpr (Cfg::EPI_BUFS > 0) {
    if (rc == GEMM_OK)
      rc = encode_tmap_3d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, uint64_t(N), uint64_t(M),
                          1, 64, Cfg::EPI_BOX_ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    tc = ta;  // the epilogue stores straight from registers: the map is unused
  }
  if (rc != GEMM_OK) return rc;
  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.L = 1;
  p.num_m_blocks = (M + Cfg::TILE_M - 1) / Cfg::TILE_M;
  p.num_n_blocks = (N + Cfg::BN - 1) / Cfg::BN;
  p.num_k_blocks = K / Cfg::BK;
  p.total_tiles = p.num_m_blocks * p.num_n_blocks;
  p.group_m = raster_group_m(p.num_m_blocks, (long long)Cfg::TILE_M * K * 2);
  p.k_splits = 1;
  p.kb_per_split = p.num_k_blocks;
  p.scale = scale2;
  p.c_ptr = C;
  p.status = dev.status;
  p.timeout_ns = wait_timeout_ns();
  // the A-scale map is unused; pass A's map in its place
  return launch_tcgen05<Cfg, Epilogue::kScaleBF16>(ta, tcode, tc, ta, tscale, p, dev, stream);
}

int launch_gemm_w4a16_t(const void* A, const uint8_t* b_t, const uint8_t* sfb_t, float scale2,
                        void* C, int M, int N, int K, int ldb, const DeviceInfo& dev,
                        cudaStream_t stream) {
  // TMA output rows must start on 16-byte boundaries
  return (N % 8 == 0)
             ? run_w4a16_t<W4PairT>(A, b_t, sfb_t, scale2, C, M, N, K, ldb, dev, stream)
             : run_w4a16_t<W4PairTDirect>(A, b_t, sfb_t, scale2, C, M, N, K, ldb, dev, stream);
}

}  // namespace gb300

namespace gb300 {

namespace {

// Weight conversion for the two-pass form: w[n][k] = e2m1 * e4m3 (exact in
// BF16), written row-major [N][K].  One thread per 32 weights (16 code
// bytes, 2 scale bytes -> 64 output bytes); consecutive threads take
// consecutive 32-weight chunks of a row.
__global__ void __launch_bounds__(256)
    w4a16_convert_kernel(const uint8_t* __restrict__ b, const uint8_t* __restrict__ sfb,
                         uint16_t* __restrict__ w, size_t chunks, int K) {
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  const size_t per_row = size_t(K) / 32;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < chunks; i += stride) {
    const size_t n = i / per_row, c = i - n * per_row;
    const uint4 codes = __ldg(reinterpret_cast<const uint4*>(b) + i);
    const uint16_t sc = __ldg(reinterpret_cast<const unsigned short*>(sfb + n * (K / 16)) + c);
    uint32_t v[16];
    w4_dequant32(codes, sc, v);
    uint4* dst = reinterpret_cast<uint4*>(w + n * size_t(K) + c * 32);
#pragma unroll
    for (int j = 0; j < 4; ++j) dst[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
}

}  // namespace

// Two-pass W4A16: convert the weights once into ws ([N][K] BF16), then the
// dense CTA-pair GEMM with the same tiles, K order and epilogue as the
// fused kernel (bit-identical results).  For large M the conversion is paid
// once instead of once per M block.
int launch_gemm_w4a16_twopass(const void* A, const uint8_t* b, const uint8_t* sfb, float scale2,
                              void* C, uint16_t* ws, int M, int N, int K, const DeviceInfo& dev,
                              cudaStream_t stream) {
  const size_t chunks = size_t(N) * size_t(K) / 32;
  const size_t want = (chunks + 255) / 256;
  const int grid = int(std::max<size_t>(1, std::min<size_t>(want, size_t(dev.num_sms) * 16)));
  w4a16_convert_kernel<<<grid, 256, 0, stream>>>(b, sfb, ws, chunks, K);
  if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
  return launch_gemm_bf16_scale(A, ws, C, M, N, K, scale2, dev, stream);
}

}  // namespace gb300
