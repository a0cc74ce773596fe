// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   C[l][m][n] = epilogue( sum_k A[l][m][k] * B[l][n][k] )      (NT layout)
//
// Operands: BF16 (kind::f16), packed e2m1 with e4m3 block scales
// (kind::mxf4nvf4, scale_vec::4X), or BF16 A with packed e2m1 B converted
// to BF16 on chip (W4A16, kind::f16).  A CTA group (one CTA, or a pair of
// CTAs on two SMs running cta_group::2 MMAs) walks the output tiles
// tile = cluster + i * clusters in grouped-M raster order (seg_at: also the
// split-K and stream-K schedules).  A tile is (128 * CG) x BN; each CTA
// stages its own 128 rows of A and BN/CG rows of B.
// Roles per CTA:
//   warp 0        TMA producer: A/B tiles (128-byte swizzle) and, for NVFP4,
//                 the 512-byte scale atoms, into a STAGES-deep smem ring;
//   warp 1        allocates TMEM; lane 0 of the leader CTA issues the MMAs
//                 (and, for NVFP4, tcgen05.cp's each stage's scale atoms
//                 into a per-stage TMEM slot first);
//   warps 2..     epilogue: tcgen05.ld -> convert (bf16 / fp16 / scaled-acc)
//                 -> swizzled smem box -> TMA store; for scaled-acc the old
//                 output box is TMA-loaded into the same smem first.  With 8
//                 epilogue warps and a single TMEM accumulator
//                 ("register-staged") every accumulator column is read into
//                 registers before the accumulator is released, so the
//                 epilogue still overlaps the next tile's MMAs; with two
//                 accumulators 8 warps take half of the columns each;
//   W4A16 only    8 conversion warps (packed codes -> BF16 B stages) and
//                 one warp TMA-loading the codes and scales into a ring.
// Every wait is bounded (globaltimer); a timeout records a code in the
// device status word, raises a CTA-wide abort flag, drains in-flight copies
// and MMAs, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "epilogue_math.cuh"
#include "ptx.cuh"
#include "watchdog.cuh"

namespace gb300 {

enum class Operand : int { kBF16 = 0, kNVFP4 = 1, kW4A16 = 2 };
// kScaleBF16: C = bf16(scale * acc), one FP32 multiply then one rounding
enum class Epilogue : int {
  kStoreBF16 = 0,
  kScaledAccBF16 = 1,
  kStoreFP16 = 2,
  kStoreF32 = 3,
  kScaleBF16 = 4
};

struct GemmParams {
  int M, N, K, L;                 // K in elements
  int num_m_blocks, num_n_blocks, num_k_blocks, total_tiles;
  int rest_m, rest_n, rest_k;     // NVFP4 scale layout extents: M/128, N/128, K/64
  int k_splits, kb_per_split;     // split-K: batch slot l = batch * k_splits + split; the
                                  // split selects K blocks [split*kb_per_split, +kb_per_split);
                                  // 1 / num_k_blocks otherwise
  float scale;                    // scaled-acc factor
  void* c_ptr;                    // output base (direct-store epilogue only)
  unsigned int* status;           // device status word
  unsigned long long timeout_ns;  // bound on every wait
  int group_m;                    // M blocks per raster group (raster_group_m)
  int sk;                         // stream-K: clusters sharing the tail (0 = off)
};

template <Operand OP, int CG_, int BN_, int STAGES_, int EPI_WARPS_ = 4, int EPI_BUFS_ = 2,
          bool SFA_REP_ = true, bool SFB_REP_ = false, int KSUB_ = 1, bool B_MN_ = false,
          bool C_T_ = false>
struct TileCfg {
  static constexpr Operand kOp = OP;
  static constexpr bool kFP4 = (OP == Operand::kNVFP4);
  // W4A16: BF16 MMAs whose B operand (NVFP4 weights) is dequantised into the
  // stage by dedicated warps instead of being loaded by TMA.
  static constexpr bool kW4 = (OP == Operand::kW4A16);
  static constexpr int CG = CG_;                  // CTAs per MMA (1 or 2)
  static constexpr int CLUSTER = CG;              // CTAs per cluster: the MMA's CTA group
  static constexpr int BM = 128;                  // A rows / TMEM lanes per CTA
  static constexpr int TILE_M = BM * CG;          // C rows per tile
  static constexpr int BN = BN_;                  // C columns per tile (MMA N)
  static constexpr int B_ROWS = BN / CG;          // B rows staged per CTA
  static constexpr int STAGES = STAGES_;
  static constexpr int EPI_WARPS = EPI_WARPS_;
  static constexpr int EPI_BUFS = EPI_BUFS_;
  static constexpr int EPI_COLS = BN / (EPI_WARPS / 4);  // accumulator columns per epilogue warp
  // KSUB = 2 (BF16): a stage holds two 64-deep K sub-tiles per operand (two
  // TMA boxes each), i.e. 8 MMAs per stage.  The per-stage work of the MMA
  // issuer (barrier probe, release commit, bookkeeping) then has 1024 pipe
  // cycles to hide behind instead of 512.
  static constexpr int KSUB = KSUB_;
  // B_MN: B is stored [K][N] (N contiguous, the NN layout).  Each stage holds
  // the CTA's B columns as 64-column atoms (BK rows of 128 bytes each, the
  // TMA's 128-byte swizzle), and the MMA reads B MN-major.
  static constexpr bool B_MN = B_MN_;
  // C_T: the output is D transposed (the swapped-operand decode GEMM, whose
  // M role holds the weights and N role the few activation rows)
  static constexpr bool C_T = C_T_;
  static constexpr int BK = kFP4 ? 256 : 64 * KSUB;  // K elements per stage
  static constexpr int KX = kFP4 ? 128 : 64;      // TMA x-extent per sub-tile (bytes or elements)
  static constexpr int MMA_K = kFP4 ? 64 : 16;    // K per MMA = 32 bytes per row
  static constexpr int KSTEPS = BK / MMA_K;       // 4 MMAs per stage
  static constexpr int A_SUB_BYTES = BM * 128;      // one 128-byte-wide K sub-tile
  static constexpr int B_SUB_BYTES = B_ROWS * 128;
  static constexpr int A_BYTES = A_SUB_BYTES * KSUB;
  static constexpr int B_BYTES = B_SUB_BYTES * KSUB;
  static constexpr int SF_ATOM = 512;             // 128 rows x 4 scales
  static constexpr int SFB_ATOMS = kFP4 ? BN / 128 : 0;  // every CTA holds the scales of all BN rows of B
  // NVFP4 scale staging for A.  The block-scaled MMA reads the four scales
  // of row 32*i + g from TMEM lane 32*i + g, column base + i; the replicating
  // 32x128b copy writes every 512-byte atom into all four lane quarters.
  // With SFA_REP each atom is instead staged four times in shared memory
  // (one replica per lane quarter) so that one 128-lane x 32-byte copy fills
  // the scale columns of two MMAs: 2 copies per stage instead of 4 (the
  // tensor pipe slows down sharply past ~10 copies per 4-MMA stage).
  static constexpr bool SFA_REP = kFP4 && SFA_REP_;
  static constexpr int SFA_BYTES = kFP4 ? KSTEPS * SF_ATOM * (SFA_REP ? 4 : 1) : 0;
  // SFB_REP: the same for B: per MMA, the 2 atoms of a 256-row B tile are
  // staged 4 times each and one 128-lane x 32-byte copy fills its 8 columns.
  static constexpr bool SFB_REP = kFP4 && SFB_REP_;
  static_assert(!SFB_REP || SFB_ATOMS == 2, "replicated B scales assume a 256-row B tile");
  static constexpr int SFB_ATOM_BYTES = kFP4 ? KSTEPS * SF_ATOM * (SFB_REP ? 4 : 1) : 0;  // per B atom
  static constexpr int SFB_BYTES = SFB_ATOMS * SFB_ATOM_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  // Output boxes: 32 rows x 64 16-bit values, or 16 rows for W4A16, whose
  // stages and code ring leave room for only 8 KB of boxes (its warps then
  // write their 32 rows as two boxes)
  static constexpr int EPI_BOX_ROWS = kW4 ? 16 : 32;
  static constexpr int EPI_BOX_BYTES = EPI_BOX_ROWS * 128;
  static constexpr int EPI_BYTES = EPI_WARPS * EPI_BUFS * EPI_BOX_BYTES;  // 0: direct stores
  // TMEM columns: accumulators first, then one scale slot per smem stage.
  static constexpr int SF_COLS = kFP4 ? KSTEPS * 4 * (1 + SFB_ATOMS) : 0;
  static constexpr int NUM_ACC = (2 * BN + STAGES * SF_COLS <= 512) ? 2 : 1;
  static constexpr int SF_TMEM_BASE = NUM_ACC * BN;
  // 8 epilogue warps with a single accumulator ("register-staged"): every
  // accumulator column is read into registers before the accumulator is
  // released; with two accumulators 8 warps split the columns in halves
  static constexpr bool kRegEpi = (EPI_WARPS == 8) && (NUM_ACC == 1);
  static constexpr int TMEM_COLS = 512;
  static_assert(NUM_ACC * BN + STAGES * SF_COLS <= TMEM_COLS, "TMEM column budget");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(CG == 1 || CG == 2, "CTA group");
  static_assert(KSUB == 1 || (KSUB == 2 && !kFP4), "K sub-tiles: BF16 only");
  static_assert(!B_MN || (!kFP4 && B_ROWS % 64 == 0), "MN-major B: BF16 operands");
  static constexpr int B_ATOM_BYTES = 64 * KSUB * 128;  // one 64-column MN-major atom of a stage
  static_assert(STAGES >= 1, "pipeline stages");
  static_assert(B_ROWS % 8 == 0, "B rows per CTA");
  static_assert(!kFP4 || BN % 128 == 0, "NVFP4 BN must cover whole 128-row scale atoms");
  static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "epilogue warps");
  static_assert(EPI_COLS % 64 == 0, "epilogue columns per warp");
  static_assert(NUM_ACC == 2 || kRegEpi, "a single accumulator needs the register-staged epilogue");
  // NVFP4: dedicated warps move each stage's scale atoms into TMEM and
  // signal sf_full[stage]; the MMA thread then issues only MMAs (every
  // tcgen05 instruction costs the issuing thread about 60 cycles).  The
  // SF_WARPS warps share every stage: warp w copies the scales of MMAs
  // [w * KSTEPS / SF_WARPS, (w + 1) * KSTEPS / SF_WARPS) and arrives on
  // sf_full[stage], which expects all of them.  A stage whose TMA data lands
  // just in time thus waits for half of its copies' issue time (6 of the 12
  // copies with unreplicated A scales take a thread about 410 cycles).
  static constexpr int SF_WARPS = kFP4 ? 2 : 0;
  static_assert(!kFP4 || (KSTEPS % (2 * SF_WARPS) == 0), "scale copies: whole MMA pairs per warp");
  static constexpr bool SF_WARP = SF_WARPS > 0;
  // W4A16: a producer warp of each CTA (RAW_WARP) TMA-loads its B rows'
  // packed codes (64 bytes per row per 128-deep K block) and block scales
  // (16 bytes per row: the scales of the even/odd pair of K blocks holding
  // the block) into a RAW_STAGES-deep ring of its own, running ahead of the
  // B stages; DQ_WARPS warps turn each job's codes into BF16 in the B stage
  // and signal bq_full[stage] on the leader CTA (every warp of both CTAs
  // arrives).  raw_full / raw_empty pace the ring.
  //
  // W4A16 with B_MN (the transposed weight layout: codes stored as K/2 rows
  // of packed bytes, byte (j, n) = elements 2j and 2j+1 of column n; scales
  // as K/16 rows): a job's codes are one 64-row x B_ROWS-byte box, its
  // scales one 8-row box, and the conversion warps write the weights
  // MN-major (64-column atoms, one 128-byte row per k), the layout the NN
  // GEMM's TMA produces.
  static constexpr bool kW4T = kW4 && B_MN;
  static constexpr int DQ_WARPS = kW4 ? 8 : 0;
  static constexpr int DQ_ROWS = kW4 ? B_ROWS / DQ_WARPS : 0;
  static constexpr int RAW_STAGES = kW4 ? 2 : 0;
  static constexpr int RAW_CODE_BYTES = kW4 ? B_ROWS * 64 : 0;  // codes of a job
  static constexpr int RAW_BYTES = kW4 ? B_ROWS * (64 + 16) : 0;  // + the scale pairs
  static constexpr int RAW_TX_BYTES = kW4T ? B_ROWS * (64 + 8) : RAW_BYTES;  // bytes a job loads
  static constexpr int RAW_RING_BYTES = RAW_STAGES * RAW_BYTES;
  static_assert(!kW4 || (KSUB == 2 && DQ_ROWS % 8 == 0 && B_ROWS <= 256),
                "W4A16: 128-deep stages");
  static_assert(!kW4T || B_ROWS == 128, "transposed W4A16: 8 column groups of 16 per CTA");
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2], epi[W][B], mma_done,
  // sf_full[S] (NVFP4) or bq_full[S], raw_full[R], raw_empty[R] (W4A16)
  static constexpr int NUM_BARS = 2 * STAGES + 4 + EPI_WARPS * EPI_BUFS + 1 +
                                  (SF_WARP ? STAGES : 0) + (kW4 ? STAGES + 2 * RAW_STAGES : 0);
  static constexpr int BAR_BYTES = NUM_BARS * 8 + 16;
  static constexpr int SMEM_BYTES =
      1024 + STAGES * STAGE_BYTES + EPI_BYTES + RAW_RING_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget (227 KB per CTA)");
  // W4A16: the warp that issues the code / scale loads
  static constexpr int RAW_WARP = kW4 ? 2 + EPI_WARPS + DQ_WARPS : -1;
  static constexpr int THREADS =
      64 + 32 * EPI_WARPS + 32 * SF_WARPS + 32 * DQ_WARPS + (kW4 ? 32 : 0);

  // Instruction descriptor.  kind::f16: D=F32 (bits 4-5 = 1), A=B=BF16
  // (bits 7-9 = 1, 10-12 = 1), both K-major, N>>3 in bits 17-22, M>>4 in
  // bits 24-28.  kind::mxf4nvf4: A=B=E2M1 (1), scale type UE4M3 (bit 23 = 0),
  // scale ids 0, dense K=64.
  __host__ __device__ static constexpr uint32_t idesc() {
    return kFP4 ? ((1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
                   (uint32_t(TILE_M >> 4) << 24))
                : ((1u << 4) | (1u << 7) | (1u << 10) | (B_MN ? (1u << 16) : 0u) |
                   (uint32_t(BN >> 3) << 17) |
                   (uint32_t(TILE_M >> 4) << 24));
  }
};

// Work item `tile` -> batch l, M block mb and N block nb, in grouped-M
// raster order: consecutive items walk group_m M blocks down one N column.
template <class Cfg>
__host__ __device__ __forceinline__ void decode_tile(int tile, const GemmParams& p, int& l,
                                                     int& mb, int& nb) {
  const int per_batch = p.num_m_blocks * p.num_n_blocks;
  l = tile / per_batch;
  const int t = tile - l * per_batch;
  const int group_tiles = p.group_m * p.num_n_blocks;
  const int g = t / group_tiles;
  const int first_m = g * p.group_m;
  const int gm = (p.num_m_blocks - first_m < p.group_m) ? p.num_m_blocks - first_m : p.group_m;
  const int r = t - g * group_tiles;
  mb = first_m + r % gm;
  nb = r / gm;
}

// One work segment of a cluster: K blocks [kb0, kb1) of tile `tile`; slot
// -1 = the whole tile (stored to C), 0 / 1 = a partial tile written as FP32
// to the cluster's stream-K workspace slot (its first / last segment).
struct Seg {
  int tile, kb0, kb1, slot;
};

// Segment `idx` of cluster c among C clusters; false past the end.  Every
// role of the kernel walks this same sequence.
//  * plain / split-K: tile = c + idx*C; with split-K the batch slot of the
//    tile selects its K blocks.
//  * stream-K (p.sk = P): the first floor(tiles/C) rounds are whole tiles
//    (tile = c + idx*C); the K iterations of the remaining tiles (the tail)
//    are split evenly over clusters 0..P-1, cluster c taking iterations
//    [T*c/P, T*(c+1)/P) in order, which makes at most its first and last
//    segment partial.
template <class Cfg>
__device__ __forceinline__ bool seg_at(const GemmParams& p, int c, int C, int idx, Seg& s) {
  if (!p.sk) {
    const long long t = (long long)c + (long long)idx * C;
    if (t >= p.total_tiles) return false;
    s.tile = int(t);
    s.slot = -1;
    s.kb0 = 0;
    s.kb1 = p.num_k_blocks;
    if (p.k_splits > 1) {
      int l, mb, nb;
      decode_tile<Cfg>(s.tile, p, l, mb, nb);
      s.kb0 = (l % p.k_splits) * p.kb_per_split;
      s.kb1 = min(p.num_k_blocks, s.kb0 + p.kb_per_split);
    }
    return true;
  }
  const int dp_rounds = p.total_tiles / C;
  if (idx < dp_rounds) {
    s.tile = c + idx * C;
    s.kb0 = 0;
    s.kb1 = p.num_k_blocks;
    s.slot = -1;
    return true;
  }
  if (c >= p.sk) return false;
  const long long kbt = p.num_k_blocks;
  const long long T = (long long)(p.total_tiles - dp_rounds * C) * kbt;
  const long long x0 = T * c / p.sk, x1 = T * (c + 1) / p.sk;
  const int j = idx - dp_rounds;
  const long long t = x0 / kbt + j;
  const long long ts = t * kbt;  // first tail iteration of tail tile t
  const long long lo = (j == 0) ? x0 : ts;
  if (lo >= x1) return false;
  const long long hi = min(x1, ts + kbt);
  s.tile = dp_rounds * C + int(t);
  s.kb0 = int(lo - ts);
  s.kb1 = int(hi - ts);
  s.slot = (s.kb0 == 0 && s.kb1 == kbt) ? -1 : (j == 0 ? 0 : 1);
  return true;
}

// Converts 8 accumulator columns (v[0..7], FP32 bits) of one row and the
// row's previous 8 output values (scaled-acc only) into one 16-byte chunk.
template <Epilogue EPI>
__device__ __forceinline__ uint4 epi_chunk(const uint32_t* v, uint4 old, float scale) {
  uint4 o;
  if constexpr (EPI == Epilogue::kStoreBF16) {
    o.x = pack_bf16x2(v[0], v[1]);
    o.y = pack_bf16x2(v[2], v[3]);
    o.z = pack_bf16x2(v[4], v[5]);
    o.w = pack_bf16x2(v[6], v[7]);
  } else if constexpr (EPI == Epilogue::kScaleBF16) {
    uint32_t* q = &o.x;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      q[i] = pack_bf16x2(__float_as_uint(__fmul_rn(scale, __uint_as_float(v[2 * i]))),
                         __float_as_uint(__fmul_rn(scale, __uint_as_float(v[2 * i + 1]))));
  } else if constexpr (EPI == Epilogue::kScaledAccBF16) {
    o.x = scaled_acc_bf16x2(old.x, pack_bf16x2(v[0], v[1]), scale);
    o.y = scaled_acc_bf16x2(old.y, pack_bf16x2(v[2], v[3]), scale);
    o.z = scaled_acc_bf16x2(old.z, pack_bf16x2(v[4], v[5]), scale);
    o.w = scaled_acc_bf16x2(old.w, pack_bf16x2(v[6], v[7]), scale);
  } else {
    o.x = pack_f16x2(v[0], v[1]);
    o.y = pack_f16x2(v[2], v[3]);
    o.z = pack_f16x2(v[4], v[5]);
    o.w = pack_f16x2(v[6], v[7]);
  }
  return o;
}

// Writes 64 converted columns of this lane's row into a 32-row x 128-byte
// box laid out with the 128-byte swizzle (16-byte chunk j of row r at
// position j ^ (r % 8)), which is what the TMA store expects.
template <Epilogue EPI>
__device__ __forceinline__ void write_box_row(uint8_t* row, int lane, const uint32_t (&lo)[32],
                                              const uint32_t (&hi)[32], float scale) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4* chunk = reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4));
    uint4 old = make_uint4(0, 0, 0, 0);
    if constexpr (EPI == Epilogue::kScaledAccBF16) old = *chunk;
    *chunk = epi_chunk<EPI>(&lo[8 * j], old, scale);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4* chunk = reinterpret_cast<uint4*>(row + (((j + 4) ^ (lane & 7)) << 4));
    uint4 old = make_uint4(0, 0, 0, 0);
    if constexpr (EPI == Epilogue::kScaledAccBF16) old = *chunk;
    *chunk = epi_chunk<EPI>(&hi[8 * j], old, scale);
  }
}

// FP32 partials: 32 accumulator columns of this lane's row = one 128-byte
// box row (4 values per 16-byte chunk), same swizzle.
__device__ __forceinline__ void write_box_row_f32(uint8_t* row, int lane, const uint32_t (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4* chunk = reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4));
    *chunk = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
}

// W4A16 weights ("gemm_dense.rs", w4a16_gemm: C = A @ dequant(B), NVFP4
// weights dequantised to BF16): 16 packed bytes of one weight row (32 e2m1
// codes, element 2j in the low nibble of byte j) and the row's two e4m3
// block scales for those elements (low byte: elements 0..15) ->
//   w = e2m1 * e4m3
// as 16 bf16x2 words in element order.  The product has at most six
// significant bits and lies in [2^-10, 2688], so BF16 holds it exactly and
// the BF16 multiply below rounds nothing (the per-tensor scale is applied
// to the FP32 sum in the epilogue).
//
// The e2m1 code -> BF16 step is a byte-permute table lookup (integer pipe):
// the magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 of codes 0..7 are the BF16
// patterns 0x0000 3F00 3F80 3FC0 4000 4040 4080 40C0; one PRMT looks up the
// low bytes of four codes, one the high bytes, and the code's sign bit
// (bit 3) becomes bit 15 of its BF16 value.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four e2m1 codes (the low 16 bits of g, code i in bits 4i..4i+3) -> two
// bf16x2 words (codes 0, 1 and codes 2, 3).
__device__ __forceinline__ void e2m1x4_to_bf16(uint32_t g, uint32_t& w01, uint32_t& w23) {
  constexpr uint32_t kLo0 = 0xC0800000u, kLo1 = 0xC0804000u;  // low bytes, codes 0..3 / 4..7
  constexpr uint32_t kHi0 = 0x3F3F3F00u, kHi1 = 0x40404040u;  // high bytes
  const uint32_t sel = g & 0x7777u;
  const uint32_t lo = prmt(kLo0, kLo1, sel);
  uint32_t hi = prmt(kHi0, kHi1, sel);
  // sign: a negative code selects byte 4 (0x80) in sign-replicate mode
  // (0xFF), a positive one byte 4 as is (0x80); bit 6 then says which
  const uint32_t sg = prmt(0u, 0x80u, (g & 0x8888u) | 0x4444u);
  hi |= (sg << 1) & 0x80808080u;  // bit 7 of a byte: bit 6 of its sg byte
  w01 = prmt(lo, hi, 0x5140u);
  w23 = prmt(lo, hi, 0x7362u);
}

// The same lookup for the transposed layout, where a byte holds two k of one
// column: four codes (g: lo/hi nibble of column n, lo/hi nibble of column
// n+1) -> the bf16x2 word of (k even; n, n+1) and of (k odd; n, n+1).
__device__ __forceinline__ void e2m1x4_to_bf16_kpairs(uint32_t g, uint32_t& w_even,
                                                      uint32_t& w_odd) {
  constexpr uint32_t kLo0 = 0xC0800000u, kLo1 = 0xC0804000u;
  constexpr uint32_t kHi0 = 0x3F3F3F00u, kHi1 = 0x40404040u;
  const uint32_t sel = g & 0x7777u;
  const uint32_t lo = prmt(kLo0, kLo1, sel);
  uint32_t hi = prmt(kHi0, kHi1, sel);
  const uint32_t sg = prmt(0u, 0x80u, (g & 0x8888u) | 0x4444u);
  hi |= (sg << 1) & 0x80808080u;
  w_even = prmt(lo, hi, 0x6240u);  // codes 0 and 2
  w_odd = prmt(lo, hi, 0x7351u);   // codes 1 and 3
}

// Transposed-layout W4A16 chunk: 16 code bytes (columns n0 .. n0+15 of one
// k pair 2j, 2j+1) and the 16 e4m3 scales of those columns -> the bf16
// weights of row k = 2j (ev, column pairs in order) and k = 2j+1 (od).
// Each product is exact (at most six significant bits).
__device__ __forceinline__ void w4t_dequant_chunk(const uint4 codes, const uint4 scales,
                                                  uint32_t (&ev)[8], uint32_t (&od)[8]) {
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
  const uint32_t sw[4] = {scales.x, scales.y, scales.z, scales.w};
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const uint32_t g = (cw[p >> 1] >> (16 * (p & 1))) & 0xFFFFu;
    const uint16_t s2 = uint16_t((sw[p >> 1] >> (16 * (p & 1))) & 0xFFFFu);
    uint32_t s16;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16) : "h"(s2));
    const __nv_bfloat162 sc =
        __float22bfloat162_rn(__half22float2(*reinterpret_cast<const __half2*>(&s16)));
    uint32_t we, wo;
    e2m1x4_to_bf16_kpairs(g, we, wo);
    const __nv_bfloat162 qe = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&we), sc);
    const __nv_bfloat162 qo = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&wo), sc);
    ev[p] = *reinterpret_cast<const uint32_t*>(&qe);
    od[p] = *reinterpret_cast<const uint32_t*>(&qo);
  }
}

__device__ __forceinline__ void w4_dequant32(const uint4 raw, uint16_t sc2, uint32_t (&out)[16]) {
  // the two block scales as bf16 (exact), each broadcast to both halves
  uint32_t s16;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16) : "h"(sc2));
  const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&s16));
  const __nv_bfloat162 s0 = __float2bfloat162_rn(sf.x), s1 = __float2bfloat162_rn(sf.y);
  const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t c[4];
    e2m1x4_to_bf16(wd[i] & 0xFFFFu, c[0], c[1]);
    e2m1x4_to_bf16(wd[i] >> 16, c[2], c[3]);
    const __nv_bfloat162 sc = (i < 2) ? s0 : s1;  // elements 0..15 / 16..31
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 q = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&c[j]), sc);
      out[4 * i + j] = *reinterpret_cast<const uint32_t*>(&q);
    }
  }
}

template <class Cfg, Epilogue EPI>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tcgen05_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_c,
                        const __grid_constant__ CUtensorMap tmap_sfa,
                        const __grid_constant__ CUtensorMap tmap_sfb, const GemmParams p) {
  constexpr int STAGES = Cfg::STAGES;
  constexpr int BN = Cfg::BN;
  constexpr int CG = Cfg::CG;
  constexpr bool kFP4 = Cfg::kFP4;
  // Scaled-acc with LA_SETS >= 2 sets of output boxes per epilogue warp (one
  // tile's boxes each): the old output of the next LA_SETS - 1 tiles is
  // requested before this tile's accumulator is awaited.
  constexpr int LA_NCH = Cfg::EPI_COLS / 64;  // 64-column boxes per warp and tile
  constexpr int LA_SETS = Cfg::EPI_BUFS / LA_NCH;
  constexpr bool kLookahead = (EPI == Epilogue::kScaledAccBF16) && !Cfg::kRegEpi &&
                              (Cfg::EPI_BUFS % LA_NCH == 0) && (LA_SETS >= 2);
  // Without epilogue buffers the 16-bit outputs are written straight from
  // registers with 16-byte global stores (frees shared memory for stages).
  constexpr bool kDirectStore = (Cfg::EPI_BUFS == 0);
  static_assert(!kDirectStore || EPI == Epilogue::kStoreBF16 || EPI == Epilogue::kStoreFP16 ||
                    EPI == Epilogue::kScaleBF16 ||
                    (EPI == Epilogue::kStoreF32 && (Cfg::kRegEpi || Cfg::C_T)),
                "direct stores serve the plain 16-bit epilogues and FP32 partials");
  static_assert(!Cfg::C_T || EPI == Epilogue::kStoreF32 || EPI == Epilogue::kStoreFP16,
                "transposed output: FP32 partials or FP16");
  static_assert(!Cfg::C_T || kDirectStore || Cfg::EPI_BUFS == 1,
                "transposed output through shared memory: one 32 x 32 box per warp");
  // L2 policy hints: keep the operands resident (they are re-read by other
  // tiles), let the once-written output leave first.
  constexpr bool kHintLoads = true;
  constexpr bool kL2Hints = true;  // output stores
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t epi_base = sbase + STAGES * Cfg::STAGE_BYTES;
  const uint32_t raw_base = epi_base + Cfg::EPI_BYTES;  // W4A16 code / scale ring
  const uint32_t bar_base = raw_base + Cfg::RAW_RING_BYTES;
  auto stage_a = [&](int s) { return sbase + s * Cfg::STAGE_BYTES; };
  auto stage_b = [&](int s) { return stage_a(s) + Cfg::A_BYTES; };
  auto stage_sfa = [&](int s) { return stage_b(s) + Cfg::B_BYTES; };
  auto stage_sfb = [&](int s) { return stage_sfa(s) + Cfg::SFA_BYTES; };
  auto full_bar = [&](int s) { return bar_base + 8 * s; };
  auto empty_bar = [&](int s) { return bar_base + 8 * (STAGES + s); };
  auto acc_full = [&](int b) { return bar_base + 8 * (2 * STAGES + b); };
  auto acc_empty = [&](int b) { return bar_base + 8 * (2 * STAGES + 2 + b); };
  auto epi_bar = [&](int e, int b) {
    return bar_base + 8 * (2 * STAGES + 4 + e * Cfg::EPI_BUFS + b);
  };
  const uint32_t mma_done = bar_base + 8 * (2 * STAGES + 4 + Cfg::EPI_WARPS * Cfg::EPI_BUFS);
  auto sf_full = [&](int s) { return mma_done + 8 * (1 + s); };
  auto bq_full = sf_full;  // W4A16 (which has no scale warps): B dequantised
  auto raw_full = [&](int q) { return mma_done + 8 * (1 + STAGES + q); };  // W4A16 codes landed
  auto raw_empty = [&](int q) {  // W4A16: every conversion warp has read slot q
    return mma_done + 8 * (1 + STAGES + Cfg::RAW_STAGES + q);
  };
  // the barrier that says stage s may be multiplied: its TMA data landed,
  // and (NVFP4) its scales are in TMEM, or (W4A16) its B is dequantised
  auto ready_bar = [&](int s) { return (Cfg::SF_WARP || Cfg::kW4) ? sf_full(s) : full_bar(s); };
  // W4A16: stage s may be multiplied once its A tiles landed (full) and its
  // B rows were converted (bq_full); the MMA issuer waits on both itself
  // (a chain of waits through the conversion warps would add a second
  // wake-up to every refill of the ring)
  auto ready_wait = [&](int s, uint32_t ph, const Watch& wt) {
    if constexpr (Cfg::kW4)
      return wait_bar(bq_full(s), ph, wt, 3) && wait_bar(full_bar(s), ph, wt, 3);
    else
      return wait_bar(ready_bar(s), ph, wt, 3);
  };
  uint8_t* misc = smem + (bar_base - sbase) + 8 * Cfg::NUM_BARS;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(misc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (Cfg::CLUSTER > 1) ? ptx::cluster_ctarank() : 0u;
  const uint32_t peer = (CG == 2) ? (rank & 1u) : 0u;  // role within the CTA pair
  const uint32_t pair_leader = 0u;                     // rank of the pair's MMA issuer
  const bool leader = (peer == 0);
  const int cluster_id = blockIdx.x / Cfg::CLUSTER;
  const int num_clusters = gridDim.x / Cfg::CLUSTER;
  // tcgen05.commit targets: both CTAs of the pair (stage releases and
  // accumulator hand-over)
  const uint16_t pair_mask = uint16_t(3u);
  const uint16_t release_mask = pair_mask;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);  // released by the MMA issuer's commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(acc_full(b), 1);
      ptx::mbar_init(acc_empty(b), Cfg::EPI_WARPS * CG);
    }
    for (int e = 0; e < Cfg::EPI_WARPS; ++e)
      for (int b = 0; b < Cfg::EPI_BUFS; ++b) ptx::mbar_init(epi_bar(e, b), 1);
    ptx::mbar_init(mma_done, 1);
    if constexpr (Cfg::SF_WARP)
      for (int s = 0; s < STAGES; ++s) ptx::mbar_init(sf_full(s), Cfg::SF_WARPS);
    if constexpr (Cfg::kW4) {
      for (int s = 0; s < STAGES; ++s) ptx::mbar_init(bq_full(s), Cfg::DQ_WARPS * CG);
      for (int q = 0; q < Cfg::RAW_STAGES; ++q) {
        ptx::mbar_init(raw_full(q), 1);
        ptx::mbar_init(raw_empty(q), Cfg::DQ_WARPS);
      }
    }
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  // The producer's first segment, found before the dependency wait: the
  // schedule arithmetic run for the first time cost ~0.7 us between the
  // wait and the first load.
  Seg s0{};
  int l0 = 0, mb0 = 0, nb0 = 0;
  bool has0 = false;
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_a);
    ptx::prefetch_tmap(&tmap_b);
    ptx::prefetch_tmap(&tmap_c);
    if constexpr (kFP4) {
      ptx::prefetch_tmap(&tmap_sfa);
      ptx::prefetch_tmap(&tmap_sfb);
    } else if constexpr (Cfg::kW4) {
      ptx::prefetch_tmap(&tmap_sfb);  // the block scales (tmap_b: the codes)
    } else if (p.sk) {
      ptx::prefetch_tmap(&tmap_sfa);  // the stream-K workspace
    }
    {
      // The operand tiles of this CTA's first stages are pulled into L2
      // while the previous grid on the stream finishes.  A prefetch moves
      // no data into the CTA, so it may come before griddepcontrol.wait;
      // the loads that follow it read the coherent L2 whatever the
      // previous grid wrote.
      has0 = seg_at<Cfg>(p, cluster_id, num_clusters, 0, s0);
      if (has0) {
        decode_tile<Cfg>(s0.tile, p, l0, mb0, nb0);
        const int l = (p.k_splits > 1) ? l0 / p.k_splits : l0;
        const int a_row = mb0 * Cfg::TILE_M + int(peer) * Cfg::BM;
        const int b_row = nb0 * BN + int(peer) * Cfg::B_ROWS;
        const int kend = min(s0.kb1, s0.kb0 + STAGES);
        for (int kb = s0.kb0; kb < kend; ++kb) {
#pragma unroll
          for (int sub = 0; sub < Cfg::KSUB; ++sub) {
            const int x = kb * Cfg::KX * Cfg::KSUB + sub * Cfg::KX;
            ptx::tma_prefetch_3d(&tmap_a, x, a_row, l);
            if constexpr (!Cfg::kW4 && !Cfg::B_MN) ptx::tma_prefetch_3d(&tmap_b, x, b_row, l);
          }
          if constexpr (kFP4 && Cfg::SFA_REP)
            ptx::tma_prefetch_3d(&tmap_sfa, 0, 0,
                                 (l * p.rest_m + mb0 * CG + int(peer)) * p.rest_k + 4 * kb);
        }
      }
    }
    // The next grid on the stream (the split-K reduce, the stream-K fixup,
    // or the next GEMM) may be scheduled now: it waits for this grid's end
    // before it touches global memory.
    ptx::griddep_launch_dependents();
  }
  if (warp == 1) {
    ptx::tmem_alloc<CG>(ptx::smem_u32(const_cast<uint32_t*>(tmem_slot)), Cfg::TMEM_COLS);
    ptx::tmem_relinquish<CG>();
  }
  ptx::tc_fence_before();
  if constexpr (Cfg::CLUSTER > 1) ptx::cluster_sync(); else __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const Watch w{abort_flag, p.status, p.timeout_ns};
  // launched as a programmatic dependent: the previous grid on the stream
  // must be complete (and its writes visible) before any global access
  ptx::griddep_wait();

  // NVFP4: the scale atoms of MMA j of stage s go into the stage's TMEM
  // slot (issued by the scale warp, which then commits sf_full[s]).
  // Descriptors and TMEM addresses of stage 0; stage s adds
  // s * STAGE_BYTES >> 4 to a descriptor's start field (no carry, as
  // for the operand descriptors) and s * SF_COLS to a TMEM column.
  const uint32_t sf_t0 = tmem_base + uint32_t(Cfg::SF_TMEM_BASE);
  uint64_t sfa_d0 = 0, sfb_d0 = 0;
  if constexpr (kFP4) {
    sfa_d0 = Cfg::SFA_REP ? ptx::smem_desc(stage_sfa(0), 4 * Cfg::SF_ATOM, 128, 0)
                          : ptx::smem_desc(stage_sfa(0), 0, 128, 0);
    sfb_d0 = Cfg::SFB_REP ? ptx::smem_desc(stage_sfb(0), Cfg::SFB_ATOM_BYTES, 128, 0)
                          : ptx::smem_desc(stage_sfb(0), 0, 128, 0);
  }
  auto copy_scales_for = [&](uint32_t sfa_t, uint64_t soff, int j) {
    if constexpr (kFP4) {
      const uint32_t sfb_t = sfa_t + Cfg::KSTEPS * 4;
      if constexpr (Cfg::SFA_REP) {
        // replicas of atoms j and j+1 -> lanes 0..127, columns 4j .. 4j+7
        if (j % 2 == 0)
          ptx::tc_cp_128x256b<CG>(sfa_t + 4 * j,
                                  sfa_d0 + soff + uint64_t((4 * j * Cfg::SF_ATOM) >> 4));
      } else {
        ptx::tc_cp_32x128b_warpx4<CG>(sfa_t + 4 * j,
                                      sfa_d0 + soff + uint64_t((j * Cfg::SF_ATOM) >> 4));
      }
      if constexpr (Cfg::SFB_REP) {
        // replicas of B atom 0 (columns +0..3) and atom 1 (+4..7)
        ptx::tc_cp_128x256b<CG>(sfb_t + 8 * j,
                                sfb_d0 + soff + uint64_t((4 * j * Cfg::SF_ATOM) >> 4));
      } else {
#pragma unroll
        for (int at = 0; at < Cfg::SFB_ATOMS; ++at)
          ptx::tc_cp_32x128b_warpx4<CG>(
              sfb_t + j * 4 * Cfg::SFB_ATOMS + 4 * at,
              sfb_d0 + soff + uint64_t(((at * Cfg::KSTEPS + j) * Cfg::SF_ATOM) >> 4));
      }
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_ab = ptx::policy_evict_last();
      (void)pol_ab;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;  // bit s: stage s has a load in flight / its parity
      bool ok = true;
      Seg sg;
      for (int idx = 0; ok; ++idx) {
        int l, mb, nb;
        if (idx == 0) {
          if (!has0) break;
          sg = s0;
          l = l0;
          mb = mb0;
          nb = nb0;
        } else {
          if (!seg_at<Cfg>(p, cluster_id, num_clusters, idx, sg)) break;
          decode_tile<Cfg>(sg.tile, p, l, mb, nb);
        }
        const int a_row = mb * Cfg::TILE_M + int(peer) * Cfg::BM;
        const int b_row = nb * BN + int(peer) * Cfg::B_ROWS;
        int sfb_atoms = 0;
        if constexpr (kFP4) sfb_atoms = min(Cfg::SFB_ATOMS, p.rest_n - nb * Cfg::SFB_ATOMS);
        const uint32_t tx =
            uint32_t(CG) * (Cfg::A_BYTES + (Cfg::kW4 ? 0 : Cfg::B_BYTES) + Cfg::SFA_BYTES +
                            uint32_t(sfb_atoms) * Cfg::SFB_ATOM_BYTES);
        // split-K: the batch slot holds batch * k_splits + split
        const int kb_begin = sg.kb0;
        const int kb_end = sg.kb1;
        if (p.k_splits > 1) l = l / p.k_splits;
        for (int kb = kb_begin; kb < kb_end; ++kb) {
          if (!wait_bar(empty_bar(stage), phase ^ 1u, w, 1)) {
            ok = false;
            break;
          }
          if (leader) ptx::mbar_arrive_expect_tx(full_bar(stage), tx);
          if constexpr (CG == 1) {
            const uint32_t fb = full_bar(stage);
#pragma unroll
            for (int sub = 0; sub < Cfg::KSUB; ++sub) {
              const int x = kb * Cfg::KX * Cfg::KSUB + sub * Cfg::KX;
              const uint32_t da = stage_a(stage) + sub * Cfg::A_SUB_BYTES;
              const uint32_t db = stage_b(stage) + sub * Cfg::B_SUB_BYTES;
              if constexpr (Cfg::kW4) {
                (void)db;
                ptx::tma_load_3d_hint(da, &tmap_a, fb, x, a_row, l, pol_ab);
              } else if constexpr (Cfg::B_MN) {
                // B [K][N]: 64-column atoms of all BK rows, loaded once per stage
                ptx::tma_load_3d_hint(da, &tmap_a, fb, x, a_row, l, pol_ab);
                if (sub == 0)
#pragma unroll
                  for (int at = 0; at < Cfg::B_ROWS / 64; ++at)
                    ptx::tma_load_3d_hint(stage_b(stage) + at * Cfg::B_ATOM_BYTES, &tmap_b, fb,
                                          b_row + 64 * at, kb * Cfg::BK, l, pol_ab);
              } else if constexpr (kHintLoads) {
                ptx::tma_load_3d_hint(da, &tmap_a, fb, x, a_row, l, pol_ab);
                ptx::tma_load_3d_hint(db, &tmap_b, fb, x, b_row, l, pol_ab);
              } else {
                ptx::tma_load_3d(da, &tmap_a, fb, x, a_row, l);
                ptx::tma_load_3d(db, &tmap_b, fb, x, b_row, l);
              }
            }
            if constexpr (kFP4) {
              // 4 consecutive atoms (tile_k = 4kb .. 4kb+3) = 2 KB = 256 u64 per 128 rows
              if constexpr (Cfg::SFA_REP) {
                // one box = the stage's 4 atoms, each 4 times ([atom][replica][512 B])
                ptx::tma_load_3d(stage_sfa(stage), &tmap_sfa, fb, 0, 0,
                                 (l * p.rest_m + mb) * p.rest_k + 4 * kb);
              } else {
                ptx::tma_load_3d(stage_sfa(stage), &tmap_sfa, fb, kb * 256, l * p.rest_m + mb, 0);
              }
              for (int at = 0; at < sfb_atoms; ++at) {
                if constexpr (Cfg::SFB_REP)
                  ptx::tma_load_3d(stage_sfb(stage) + at * Cfg::SFB_ATOM_BYTES, &tmap_sfb, fb, 0, 0,
                                   (l * p.rest_n + nb * Cfg::SFB_ATOMS + at) * p.rest_k + 4 * kb);
                else
                  ptx::tma_load_3d(stage_sfb(stage) + at * Cfg::KSTEPS * Cfg::SF_ATOM, &tmap_sfb,
                                   fb, kb * 256, l * p.rest_n + nb * Cfg::SFB_ATOMS + at, 0);
              }
            }
          } else {
            const uint32_t fb = ptx::mapa_shared(full_bar(stage), pair_leader);  // the leader's barrier
#pragma unroll
            for (int sub = 0; sub < Cfg::KSUB; ++sub) {
              const int x = kb * Cfg::KX * Cfg::KSUB + sub * Cfg::KX;
              const uint32_t da = stage_a(stage) + sub * Cfg::A_SUB_BYTES;
              const uint32_t db = stage_b(stage) + sub * Cfg::B_SUB_BYTES;
              if constexpr (Cfg::kW4) {
                (void)db;  // B is written by the dequantisation warps
                ptx::tma_load_3d_pair_hint(da, &tmap_a, fb, x, a_row, l, pol_ab);
              } else if constexpr (Cfg::B_MN) {
                ptx::tma_load_3d_pair_hint(da, &tmap_a, fb, x, a_row, l, pol_ab);
                if (sub == 0)
#pragma unroll
                  for (int at = 0; at < Cfg::B_ROWS / 64; ++at)
                    ptx::tma_load_3d_pair_hint(stage_b(stage) + at * Cfg::B_ATOM_BYTES, &tmap_b,
                                               fb, b_row + 64 * at, kb * Cfg::BK, l, pol_ab);
              } else if constexpr (kHintLoads) {
                ptx::tma_load_3d_pair_hint(da, &tmap_a, fb, x, a_row, l, pol_ab);
                ptx::tma_load_3d_pair_hint(db, &tmap_b, fb, x, b_row, l, pol_ab);
              } else {
                ptx::tma_load_3d_pair(da, &tmap_a, fb, x, a_row, l);
                ptx::tma_load_3d_pair(db, &tmap_b, fb, x, b_row, l);
              }
            }
            if constexpr (kFP4) {
              if constexpr (Cfg::SFA_REP) {
                ptx::tma_load_3d_pair(stage_sfa(stage), &tmap_sfa, fb, 0, 0,
                                      (l * p.rest_m + mb * CG + int(peer)) * p.rest_k + 4 * kb);
              } else {
                ptx::tma_load_3d_pair(stage_sfa(stage), &tmap_sfa, fb, kb * 256,
                                      l * p.rest_m + mb * CG + int(peer), 0);
              }
              for (int at = 0; at < sfb_atoms; ++at) {
                if constexpr (Cfg::SFB_REP)
                  ptx::tma_load_3d_pair(
                      stage_sfb(stage) + at * Cfg::SFB_ATOM_BYTES, &tmap_sfb, fb, 0, 0,
                      (l * p.rest_n + nb * Cfg::SFB_ATOMS + at) * p.rest_k + 4 * kb);
                else
                  ptx::tma_load_3d_pair(stage_sfb(stage) + at * Cfg::KSTEPS * Cfg::SF_ATOM,
                                        &tmap_sfb, fb, kb * 256,
                                        l * p.rest_n + nb * Cfg::SFB_ATOMS + at, 0);
              }
            }
          }
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (leader) {
        // Every load issued (by either CTA of the group) must have landed
        // before the CTAs may exit: the leader's full barriers count both.
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) drain_bar(full_bar(s), (armed_parity >> s) & 1u, w);
      } else if (!ok) {
        // The peer CTA's loads complete on the leader's barriers; after an
        // abort give them time to land before this CTA can exit.
        spin_ns(2000000ull);
      }
    }
  } else if (Cfg::kW4 && warp == Cfg::RAW_WARP) {
    if (lane == 0) {
      // W4A16 codes and scales of this CTA's weight rows, job by job, into
      // the raw ring (up to RAW_STAGES jobs ahead of the conversion warps):
      // codes of K block kb, scales of the even/odd pair holding kb (the
      // 16-byte TMA box starts at an even block)
      int q = 0;
      uint32_t qphase = 0;
      uint32_t armed = 0, armed_parity = 0;
      bool ok = true;
      Seg sg;
      for (int idx = 0; ok && seg_at<Cfg>(p, cluster_id, num_clusters, idx, sg); ++idx) {
        int l, mb, nb;
        decode_tile<Cfg>(sg.tile, p, l, mb, nb);
        const int b_row = nb * BN + int(peer) * Cfg::B_ROWS;
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!wait_bar(raw_empty(q), qphase ^ 1u, w, 10)) {
            ok = false;
            break;
          }
          const uint32_t slot = raw_base + q * Cfg::RAW_BYTES;
          ptx::mbar_arrive_expect_tx(raw_full(q), Cfg::RAW_TX_BYTES);
          if constexpr (Cfg::kW4T) {
            // code rows kb*64 .. +63 and scale rows kb*8 .. +7, this CTA's
            // B_ROWS columns (x in bytes = columns)
            ptx::tma_load_3d(slot, &tmap_b, raw_full(q), b_row, kb * 64, 0);
            ptx::tma_load_3d(slot + Cfg::RAW_CODE_BYTES, &tmap_sfb, raw_full(q), b_row, kb * 8, 0);
          } else {
            ptx::tma_load_3d(slot, &tmap_b, raw_full(q), kb * 64, b_row, 0);
            ptx::tma_load_3d(slot + Cfg::RAW_CODE_BYTES, &tmap_sfb, raw_full(q), (kb & ~1) * 8,
                             b_row, 0);
          }
          armed |= 1u << q;
          armed_parity = (armed_parity & ~(1u << q)) | (qphase << q);
          if (++q == Cfg::RAW_STAGES) {
            q = 0;
            qphase ^= 1u;
          }
        }
      }
      // every load must land before the CTA may exit
      for (int r = 0; r < Cfg::RAW_STAGES; ++r)
        if (armed & (1u << r)) drain_bar(raw_full(r), (armed_parity >> r) & 1u, w);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = Cfg::idesc();
      // The tensor pipe takes the next MMA only shortly before the one it
      // is executing ends, so whatever this thread does between a stage's
      // last MMA and the next stage's first leaves the pipe idle.  The loop
      // is therefore kept to: wait for the stage (already complete when the
      // loads run ahead), fence, the stage's MMAs, the commit that releases
      // the stage.  Measured per 4-MMA stage at 4096 x 7168 x 16384 (NVFP4,
      // 649 cycles of MMA): 655 cycles median with this loop, 808 with an
      // issuer that prepared the next job between the MMAs and released a
      // stage after the next stage's first MMA (the branches around those
      // commits and probes cost more than they saved).  Tile changes
      // (accumulator hand-over, the next segment) stay outside the loop.
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // K tail: the last K block may need fewer than KSTEPS MMAs (the
      // zero-filled rest of its stage needs none)
      const int tail_kb = (p.K % Cfg::BK) ? p.K / Cfg::BK : -1;
      const int tail_steps = (p.K % Cfg::BK + Cfg::MMA_K - 1) / Cfg::MMA_K;
      // Stage s, MMA j: start address + s * STAGE_BYTES + offset of j, i.e.
      // the 14-bit start field (address >> 4) grows by that >> 4; shared
      // addresses stay below 2^18 bytes, so the field never carries over.
      const uint64_t adesc0 = ptx::sw128_kmajor_desc(stage_a(0));
      // MN-major B: leading offset = atom stride (next 64 columns), stride
      // offset = 8 K rows (1024 bytes)
      const uint64_t bdesc0 = Cfg::B_MN ? ptx::smem_desc(stage_b(0), Cfg::B_ATOM_BYTES, 1024, 2)
                                        : ptx::sw128_kmajor_desc(stage_b(0));
      Seg sg;
      int it = 0;
      for (int idx = 0; ok && seg_at<Cfg>(p, cluster_id, num_clusters, idx, sg); ++idx, ++it) {
        const int acc = it % Cfg::NUM_ACC;
        // the accumulator's previous tile must have been read by the epilogue
        if (!wait_bar(acc_empty(acc), (uint32_t(it / Cfg::NUM_ACC) & 1u) ^ 1u, w, 2)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!ready_wait(stage, phase, w)) {
            ok = false;
            break;
          }
          // scales / B written by other threads' tcgen05 copies or stores:
          // order them before the MMAs (the TMA data is ordered by the
          // full barrier itself)
          if constexpr (Cfg::SF_WARP || Cfg::kW4) ptx::tc_fence_after();
          const uint64_t soff = uint64_t(uint32_t(stage) * uint32_t(Cfg::STAGE_BYTES >> 4));
          const uint32_t sfa_t = sf_t0 + uint32_t(stage * Cfg::SF_COLS);
          const int nsteps = (kb == tail_kb) ? tail_steps : Cfg::KSTEPS;
          const bool first_kb = (kb == sg.kb0);
#pragma unroll
          for (int j = 0; j < Cfg::KSTEPS; ++j) {
            if constexpr (!Cfg::SF_WARP) copy_scales_for(sfa_t, soff, j);
            if (j < nsteps) {
              // step j: K sub-tile j / 4, 32-byte K slice j % 4 within it
              const uint64_t ad =
                  adesc0 + soff + uint64_t(((j / 4) * Cfg::A_SUB_BYTES + 32 * (j % 4)) >> 4);
              // K-major: sub-tile j / 4, 32-byte K slice j % 4; MN-major: rows 16 j ..
              const uint64_t bd =
                  Cfg::B_MN
                      ? bdesc0 + soff + uint64_t((j * 16 * 128) >> 4)
                      : bdesc0 + soff + uint64_t(((j / 4) * Cfg::B_SUB_BYTES + 32 * (j % 4)) >> 4);
              const uint32_t accum = !first_kb || (j != 0);
              if constexpr (kFP4)
                ptx::mma_nvf4<CG>(d_tmem, ad, bd, idesc, sfa_t + 4 * j,
                                  sfa_t + Cfg::KSTEPS * 4 + j * 4 * Cfg::SFB_ATOMS, accum);
              else
                ptx::mma_bf16<CG>(d_tmem, ad, bd, idesc, accum);
            }
          }
          // release the stage to both producers once these MMAs are done
          ptx::tc_commit<CG>(empty_bar(stage), release_mask);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // tile done: hand the accumulator to the epilogue
        ptx::tc_commit<CG>(acc_full(acc), pair_mask);
      }
      // Every MMA / copy issued must be complete before TMEM is released.
      ptx::tc_commit<CG>(mma_done, pair_mask);
      drain_bar(mma_done, 0, w);
    }
  } else if (Cfg::SF_WARP && warp >= 2 + Cfg::EPI_WARPS) {
    // ------------------------------------------------------------ scale copies
    // Walks the same stage sequence as the MMA issuer: once a stage's TMA
    // data has landed (which also means the MMAs that last read the
    // stage's TMEM scale slot are done: the producer refilled the stage
    // only after their release), copy this warp's share of its scale atoms
    // and commit sf_full.
    const int sfw = warp - (2 + Cfg::EPI_WARPS);
    constexpr int JPW = Cfg::KSTEPS / (Cfg::SF_WARPS > 0 ? Cfg::SF_WARPS : 1);  // MMAs per warp
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int last = -1;
      uint32_t last_phase = 0;
      bool ok = true;
      Seg sg;
      for (int idx = 0; ok && seg_at<Cfg>(p, cluster_id, num_clusters, idx, sg); ++idx) {
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!wait_bar(full_bar(stage), phase, w, 6)) {
            ok = false;
            break;
          }
          // The slot's previous readers (MMAs of the MMA thread) completed
          // before this stage could be refilled; order this thread's
          // copies after that observed completion.
          ptx::tc_fence_after();
          const uint64_t soff = uint64_t(uint32_t(stage) * uint32_t(Cfg::STAGE_BYTES >> 4));
          const uint32_t sfa_t = sf_t0 + uint32_t(stage * Cfg::SF_COLS);
#pragma unroll
          for (int j = 0; j < JPW; ++j) copy_scales_for(sfa_t, soff, sfw * JPW + j);
          ptx::tc_commit<CG>(sf_full(stage), uint16_t(1u << pair_leader));
          last = stage;
          last_phase = phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every copy must be complete before TMEM is released
      if (last >= 0) drain_bar(sf_full(last), last_phase, w);
    }
  } else if (Cfg::kW4 && warp >= 2 + Cfg::EPI_WARPS && warp < Cfg::RAW_WARP) {
    // ------------------------------------------------------------ W4A16 weights
    // Warp d owns DQ_ROWS weight rows of this CTA's half of the tile and
    // walks the same job sequence as the producers.  Per job: wait for its
    // codes and scales in the raw ring, read this warp's rows into registers,
    // wait until the MMAs that last read the B stage are done, write the
    // BF16 weights in the MMA's 128-byte-swizzled K-major layout, then one
    // fence (async proxy) orders both the raw reads and the B writes, and the
    // warp hands the raw slot back and arrives on the leader CTA's bq_full
    // (the MMA issuer also waits for the stage's A tiles on full).  Per job
    // a conversion warp measured ~730 cycles converting and ~250 in each
    // fence-and-signal, against 1298 cycles of MMA per stage, so the second
    // fence a separate early release of the raw slot needed cost more than
    // the release gained (1016 x 12288 x 2048: 49.9 -> 48.6 us).
    // Lanes: row prow (lane / 4) of an 8-row pass, K quarter kq (lane % 4).
    // The lanes of quarters 2 and 3 convert their two 16-element halves in
    // swapped order, which staggers the 16-byte chunks written together by
    // an 8-lane phase over all eight bank groups of a 128-byte row.
    if constexpr (Cfg::kW4T) {
      // Transposed weights.  A job's codes are 64 k-pair rows x 128 column
      // bytes: 512 chunks of 16 columns, two per lane.  Lane: column group
      // cq = lane % 8, k-pair row kk = pass * 32 + warp * 4 + lane / 8 (an
      // 8-lane phase reads one contiguous 128-byte row).  Each chunk gives
      // two 32-byte pieces (rows 2kk and 2kk+1) of the column group's
      // 64-column atom; lanes of the second atom write their two 16-byte
      // chunks in swapped order so that an 8-lane phase covers all eight
      // bank groups.
      constexpr int TPASSES = 64 / (Cfg::DQ_WARPS * 4);
      const int dw = warp - (2 + Cfg::EPI_WARPS);
      const int cq = lane & 7;
      const int atom = cq >> 2;
      const int c0 = (cq & 3) * 2;  // first 16-byte chunk of the group in its atom row
      const uint32_t bq_target =
          (CG == 2) ? ptx::mapa_shared(bq_full(0), pair_leader) : bq_full(0);
      int stage = 0, q = 0;
      uint32_t phase = 0, qphase = 0;
      bool ok = true;
      Seg sg;
      for (int idx = 0; ok && seg_at<Cfg>(p, cluster_id, num_clusters, idx, sg); ++idx) {
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!__all_sync(0xffffffffu, wait_bar(raw_full(q), qphase, w, 8))) {
            ok = false;
            break;
          }
          const uint8_t* slot = smem + (raw_base - sbase) + q * Cfg::RAW_BYTES;
          uint4 codes[TPASSES], scl[TPASSES];
#pragma unroll
          for (int ps = 0; ps < TPASSES; ++ps) {
            const int kk = ps * (Cfg::DQ_WARPS * 4) + dw * 4 + (lane >> 3);
            codes[ps] = *reinterpret_cast<const uint4*>(slot + kk * Cfg::B_ROWS + cq * 16);
            scl[ps] = *reinterpret_cast<const uint4*>(slot + Cfg::RAW_CODE_BYTES +
                                                      (kk >> 3) * Cfg::B_ROWS + cq * 16);
          }
          // The slot is released after the B writes below, behind the same
          // fence: it is refilled by TMA (the async proxy), which must not
          // overtake these generic reads (without a fence a load still in
          // flight at the release can return the next job's bytes).
          const int q_read = q;
          if (++q == Cfg::RAW_STAGES) {
            q = 0;
            qphase ^= 1u;
          }
          if (!__all_sync(0xffffffffu, wait_bar(empty_bar(stage), phase ^ 1u, w, 11))) {
            ok = false;
            break;
          }
          uint8_t* atom_base = smem + (stage_b(stage) - sbase) + atom * Cfg::B_ATOM_BYTES;
#pragma unroll
          for (int ps = 0; ps < TPASSES; ++ps) {
            uint32_t ev[8], od[8];
            w4t_dequant_chunk(codes[ps], scl[ps], ev, od);
            const int kk = ps * (Cfg::DQ_WARPS * 4) + dw * 4 + (lane >> 3);
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // rows 2kk (even) and 2kk+1 (odd)
              const int k = 2 * kk + h;
              const uint32_t* v = h ? od : ev;  // h is a compile-time index
              uint8_t* rowp = atom_base + k * 128;
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                // half `part` of the group (columns 0-7 / 8-15); selects keep
                // the register indices static
                const int part = i ^ atom;
                const uint4 val = atom ? make_uint4(v[4 * (1 - i)], v[4 * (1 - i) + 1],
                                                    v[4 * (1 - i) + 2], v[4 * (1 - i) + 3])
                                       : make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2],
                                                    v[4 * i + 3]);
                *reinterpret_cast<uint4*>(rowp + (((c0 + part) ^ (k & 7)) << 4)) = val;
              }
            }
          }
          // one fence orders the raw slot's generic reads (before its TMA
          // refill) and the B writes (before the tensor core reads them)
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::mbar_arrive(raw_empty(q_read));
            if constexpr (CG == 2) ptx::mbar_arrive_remote(bq_target + 8 * stage);
            else ptx::mbar_arrive(bq_full(stage));
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    } else {
    constexpr int PASSES = Cfg::kW4 ? Cfg::DQ_ROWS / 8 : 1;
    const int dw = warp - (2 + Cfg::EPI_WARPS);
    const int prow = lane >> 2;
    const int kq = lane & 3;
    const int swap = kq & 2;  // 2: halves swapped
    const uint32_t bq_target = (CG == 2) ? ptx::mapa_shared(bq_full(0), pair_leader) : bq_full(0);
    int stage = 0, q = 0;
    uint32_t phase = 0, qphase = 0;
    bool ok = true;
    Seg sg;
    for (int idx = 0; ok && seg_at<Cfg>(p, cluster_id, num_clusters, idx, sg); ++idx) {
      for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
        if (!__all_sync(0xffffffffu, wait_bar(raw_full(q), qphase, w, 8))) {
          ok = false;
          break;
        }
        const uint8_t* slot = smem + (raw_base - sbase) + q * Cfg::RAW_BYTES;
        uint4 codes[PASSES];
        uint16_t scl[PASSES];
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
          const int r = dw * Cfg::DQ_ROWS + ps * 8 + prow;  // row within the CTA's B half
          uint4 c = *reinterpret_cast<const uint4*>(slot + r * 64 + kq * 16);
          uint16_t sv = *reinterpret_cast<const uint16_t*>(slot + Cfg::RAW_CODE_BYTES + r * 16 +
                                                          (kb & 1) * 8 + kq * 2);
          if (swap) {
            c = make_uint4(c.z, c.w, c.x, c.y);
            sv = uint16_t((sv >> 8) | (sv << 8));
          }
          codes[ps] = c;
          scl[ps] = sv;
        }
        // generic reads of a slot that TMA refills: released after the B
        // writes, behind the same fence
        const int q_read = q;
        if (++q == Cfg::RAW_STAGES) {
          q = 0;
          qphase ^= 1u;
        }
        if (!__all_sync(0xffffffffu, wait_bar(empty_bar(stage), phase ^ 1u, w, 11))) {
          ok = false;
          break;
        }
        const uint32_t sub_base = stage_b(stage) + (kq >> 1) * Cfg::B_SUB_BYTES;
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
          uint32_t v[16];
          w4_dequant32(codes[ps], scl[ps], v);
          const int r = dw * Cfg::DQ_ROWS + ps * 8 + prow;
          uint8_t* rowp = smem + (sub_base - sbase) + r * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = ((kq & 1) << 2) + (i ^ swap);  // 16-byte chunk of the 128-byte row
            *reinterpret_cast<uint4*>(rowp + ((c ^ (r & 7)) << 4)) =
                make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
        // one fence orders the raw slot's generic reads (before its TMA
        // refill) and the B writes (before the tensor core reads them)
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(raw_empty(q_read));
          if constexpr (CG == 2) ptx::mbar_arrive_remote(bq_target + 8 * stage);
          else ptx::mbar_arrive(bq_full(stage));
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    }
  } else if (warp >= 2 && warp < 2 + Cfg::EPI_WARPS) {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 2;          // epilogue warp index
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int col_base = (e >> 2) * Cfg::EPI_COLS;  // first accumulator column of this warp
    const uint32_t lane_off = uint32_t(q * 32) << 16;
    const uint32_t buf0 = epi_base + e * Cfg::EPI_BUFS * Cfg::EPI_BOX_BYTES;
    // the leader CTA's acc_empty barriers (the MMA issuer waits on those)
    const uint32_t ae_leader0 =
        (CG == 2) ? ptx::mapa_shared(acc_empty(0), pair_leader) : acc_empty(0);
    const uint32_t ae_leader1 =
        (CG == 2) ? ptx::mapa_shared(acc_empty(1), pair_leader) : acc_empty(1);
    const uint64_t pol_c = ptx::policy_evict_first();
    (void)pol_c;
    auto store_box = [&](uint32_t sbuf, int col0, int row0, int l) {
      if constexpr (kL2Hints) ptx::tma_store_3d_hint(&tmap_c, sbuf, col0, row0, l, pol_c);
      else ptx::tma_store_3d(&tmap_c, sbuf, col0, row0, l);
    };
    uint32_t chunk_ctr = 0;
    uint32_t epi_parity = 0;     // bit b: parity of the next wait on epi_bar(e, b)
    uint32_t epi_pending = 0;    // bit b: a load into buffer b has not been waited for
    bool ok = true;
    int it = 0;
    // The warp's TMEM reads of the accumulator are complete (waited for);
    // hand it back to the MMA issuer.  The arrive on the leader's barrier
    // uses the default (CTA-scope) release: the cluster-scope form waited
    // for this warp's TMA output stores still in flight and cost the
    // scaled-acc epilogue about 2500 cycles per tile.
    auto release_acc = [&](int acc) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 2) ptx::mbar_arrive_remote(acc == 0 ? ae_leader0 : ae_leader1);
        else ptx::mbar_arrive(acc_empty(acc));
      }
    };
    // Look-ahead loads of the old output boxes of segment s2's tile into box set `set`.
    auto prefetch_out = [&](const Seg& s2, int set) {
      if constexpr (kLookahead) {
        constexpr int NCH = LA_NCH;
        int l2, mb2, nb2;
        decode_tile<Cfg>(s2.tile, p, l2, mb2, nb2);
        const int r0 = mb2 * Cfg::TILE_M + int(peer) * Cfg::BM + q * 32;
        if (r0 >= p.M) return;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const int col0 = nb2 * BN + col_base + c * 64;
          if (col0 >= p.N) continue;
          const int b = set * NCH + c;
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(epi_bar(e, b), Cfg::EPI_BOX_BYTES);
            ptx::tma_load_3d(buf0 + b * Cfg::EPI_BOX_BYTES, &tmap_c, epi_bar(e, b), col0, r0, l2);
          }
          epi_pending |= 1u << b;
        }
      }
    };
    Seg sg;
    if constexpr (kLookahead) {
      for (int k = 0; k < LA_SETS - 1; ++k)
        if (seg_at<Cfg>(p, cluster_id, num_clusters, k, sg)) prefetch_out(sg, k);
    }
    for (int idx = 0; ok && seg_at<Cfg>(p, cluster_id, num_clusters, idx, sg); ++idx, ++it) {
      int l, mb, nb;
      decode_tile<Cfg>(sg.tile, p, l, mb, nb);
      const int acc = it % Cfg::NUM_ACC;
      const uint32_t acc_phase = uint32_t(it / Cfg::NUM_ACC) & 1u;
      if constexpr (kLookahead) {
        Seg ns;
        if (seg_at<Cfg>(p, cluster_id, num_clusters, idx + LA_SETS - 1, ns)) {
          // that tile's set last held the previous tile's boxes: their
          // stores must have read them
          if (lane == 0) ptx::bulk_wait_group_read<0>();
          __syncwarp();
          prefetch_out(ns, (it + LA_SETS - 1) % LA_SETS);
        }
      }
      ok = __all_sync(0xffffffffu, wait_bar(acc_full(acc), acc_phase, w, 4));
      if (!ok) break;
      ptx::tc_fence_after();
      const int row0 = mb * Cfg::TILE_M + int(peer) * Cfg::BM + q * 32;
      const bool rows_live = row0 < p.M;
      const uint32_t tacc = tmem_base + lane_off + uint32_t(acc * BN + col_base);

      if constexpr (Cfg::C_T) {
        // Transposed output (the swapped-operand decode GEMM: D rows are the
        // weights, D columns the activation rows), 32 columns per TMEM read.
        // FP32 split-K partials go to [split][batch][activation row][weight],
        // FP16 results to [batch][activation row][weight].
        const int gi = row0 + lane;  // weight index (output column)
        const int nbat = p.L / p.k_splits;
        const size_t slot = (EPI == Epilogue::kStoreF32)
                                ? size_t(l % p.k_splits) * nbat + size_t(l / p.k_splits)
                                : size_t(l);
        if constexpr (kDirectStore) {
          // for each column, the warp's 32 lanes store 32 consecutive
          // output elements of one activation row
#pragma unroll 1
          for (int c = 0; c < Cfg::EPI_COLS / 32; ++c) {
            uint32_t r0[32];
            ptx::tmem_ld_32x32b_x32(tacc + uint32_t(32 * c), r0);
            ptx::tmem_ld_wait_regs(r0);
            if (c == Cfg::EPI_COLS / 32 - 1) release_acc(acc);
            const int j0 = nb * BN + col_base + 32 * c;  // activation row of r0[0]
            if (gi >= p.M) continue;
#pragma unroll
            for (int t = 0; t < 32; ++t) {
              if (j0 + t >= p.N) break;
              const size_t off = (slot * p.N + size_t(j0 + t)) * size_t(p.M) + size_t(gi);
              if constexpr (EPI == Epilogue::kStoreF32)
                static_cast<uint32_t*>(p.c_ptr)[off] = r0[t];
              else
                static_cast<uint16_t*>(p.c_ptr)[off] =
                    uint16_t(pack_f16x2(r0[t], 0u) & 0xFFFFu);
            }
          }
        } else {
          // Through this warp's box in shared memory, [32 activation rows]
          // [32 weights] (row t: the warp's 32 weights for activation row
          // j0 + t; lane = weight, so each row is written conflict-free),
          // then one TMA store per 32 columns; the tensor map clips rows
          // and weights past the output.  Scattered 4-byte stores of the
          // same data took about 4 us per 128 x 128 tile.
          // The CTA's last tile (a decode CTA's only one): its MMAs, and so
          // every use of the stages, are complete, so each box takes a
          // place of its own in the stage memory and the stores go out
          // without waiting for the previous box to be read.
          constexpr uint32_t kBoxBytes = 32 * 32 * 4;
          static_assert(Cfg::EPI_WARPS * (Cfg::EPI_COLS / 32) * kBoxBytes <=
                            Cfg::STAGES * Cfg::STAGE_BYTES,
                        "the last tile's boxes fit the stage memory");
          Seg nx;
          const bool last_tile = !seg_at<Cfg>(p, cluster_id, num_clusters, idx + 1, nx);
#pragma unroll 1
          for (int c = 0; c < Cfg::EPI_COLS / 32; ++c) {
            uint32_t r0[32];
            ptx::tmem_ld_32x32b_x32(tacc + uint32_t(32 * c), r0);
            ptx::tmem_ld_wait_regs(r0);
            if (c == Cfg::EPI_COLS / 32 - 1) release_acc(acc);
            const int j0 = nb * BN + col_base + 32 * c;  // activation row of r0[0]
            if (!rows_live || j0 >= p.N) continue;       // warp-uniform
            uint32_t bsm = buf0;
            if (last_tile) {
              bsm = sbase + uint32_t(e * (Cfg::EPI_COLS / 32) + c) * kBoxBytes;
            } else {
              if (lane == 0) ptx::bulk_wait_group_read<0>();  // the box's previous store read it
              __syncwarp();
            }
            uint8_t* box = smem + (bsm - sbase);
#pragma unroll
            for (int t = 0; t < 32; ++t) {
              if constexpr (EPI == Epilogue::kStoreF32)
                reinterpret_cast<uint32_t*>(box)[t * 32 + lane] = r0[t];
              else
                reinterpret_cast<uint16_t*>(box)[t * 32 + lane] =
                    uint16_t(pack_f16x2(r0[t], 0u) & 0xFFFFu);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_3d(&tmap_c, bsm, row0, j0, int(slot));
              ptx::bulk_commit_group();
            }
          }
        }
      } else if constexpr (Cfg::kRegEpi) {
        // Read every column of this warp first, then hand the accumulator back.
        constexpr int NCH = Cfg::EPI_COLS / 64;
        uint32_t r[2 * NCH][32];
#pragma unroll
        for (int i = 0; i < 2 * NCH; ++i) ptx::tmem_ld_32x32b_x32(tacc + 32 * i, r[i]);
#pragma unroll
        for (int i = 0; i < 2 * NCH; ++i) ptx::tmem_ld_wait_regs(r[i]);
        release_acc(acc);
        if constexpr (kDirectStore && EPI == Epilogue::kStoreF32) {
          // FP32 split-K partials: 32 columns per TMEM read, eight 16-byte
          // stores per lane (N % 4 == 0 keeps every piece whole)
          // partials [split][batch][M][N]: batch slot l = batch * k_splits + split
          const int grow = row0 + lane;
          const int nbat = p.L / p.k_splits;
          const size_t slot = size_t(l % p.k_splits) * nbat + size_t(l / p.k_splits);
          if (grow < p.M) {
            float* dst = static_cast<float*>(p.c_ptr) +
                         (slot * p.M + size_t(grow)) * size_t(p.N) + nb * BN + col_base;
#pragma unroll
            for (int i = 0; i < 2 * NCH; ++i)
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (nb * BN + col_base + 32 * i + 4 * j < p.N)
                  *reinterpret_cast<uint4*>(dst + 32 * i + 4 * j) =
                      make_uint4(r[i][4 * j], r[i][4 * j + 1], r[i][4 * j + 2], r[i][4 * j + 3]);
          }
        } else if constexpr (kDirectStore) {
          const int grow = row0 + lane;
          if (grow < p.M) {
            uint16_t* dst = static_cast<uint16_t*>(p.c_ptr) +
                            (size_t(l) * p.M + size_t(grow)) * size_t(p.N) + nb * BN + col_base;
#pragma unroll
            for (int i = 0; i < 2 * NCH; ++i)
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (nb * BN + col_base + 32 * i + 8 * j < p.N)
                  *reinterpret_cast<uint4*>(dst + 32 * i + 8 * j) =
                      epi_chunk<EPI>(&r[i][8 * j], make_uint4(0, 0, 0, 0), 0.0f);
          }
        } else {
          // the CTA's last tile: each box in a place of its own in the freed
          // stage memory, no waits (as in the other epilogues)
          constexpr bool kLastInStages =
              Cfg::EPI_WARPS * NCH * Cfg::EPI_BOX_BYTES <= Cfg::STAGES * Cfg::STAGE_BYTES;
          bool last_tile = false;
          if constexpr (kLastInStages) {
            Seg nx;
            last_tile = sg.slot < 0 && !seg_at<Cfg>(p, cluster_id, num_clusters, idx + 1, nx);
          }
#pragma unroll
        for (int c = 0; c < NCH; ++c, ++chunk_ctr) {
          const int b = int(chunk_ctr % Cfg::EPI_BUFS);
          const uint32_t sbuf =
              last_tile ? sbase + uint32_t(e * NCH + c) * Cfg::EPI_BOX_BYTES
                        : buf0 + b * Cfg::EPI_BOX_BYTES;
          const int col0 = nb * BN + col_base + c * 64;
          if (!(rows_live && col0 < p.N)) continue;
          if (!last_tile) {
            if (lane == 0) {
              if constexpr (Cfg::EPI_BUFS == 1) ptx::bulk_wait_group_read<0>();
              else ptx::bulk_wait_group_read<Cfg::EPI_BUFS - 1>();
            }
            __syncwarp();
          }
          write_box_row<EPI>(smem + (sbuf - sbase) + lane * 128, lane, r[2 * c], r[2 * c + 1],
                             p.scale);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            store_box(sbuf, col0, row0, l);
            ptx::bulk_commit_group();
          }
        }
        }
      } else if constexpr (kLookahead) {
        // Scaled-acc with look-ahead: the old output boxes of this tile were
        // requested LA_SETS - 1 tiles ago, so HBM reads overlap the MMAs and
        // the stores of the tiles in between.
        constexpr int NCH = LA_NCH;
        const int set = it % LA_SETS;
#pragma unroll 1
        for (int c = 0; c < NCH; ++c) {
          const int b = set * NCH + c;
          const uint32_t sbuf = buf0 + b * Cfg::EPI_BOX_BYTES;
          const int col0 = nb * BN + col_base + c * 64;
          const bool live = rows_live && col0 < p.N;
          uint32_t r0[32], r1[32];
          const uint32_t taddr = tacc + uint32_t(c * 64);
          ptx::tmem_ld_32x32b_x32(taddr, r0);
          ptx::tmem_ld_32x32b_x32(taddr + 32, r1);
          ptx::tmem_ld_wait_regs(r0);
          ptx::tmem_ld_wait_regs(r1);
          if (c == NCH - 1) release_acc(acc);
          if (!live) continue;
          const bool got = wait_bar(epi_bar(e, b), (epi_parity >> b) & 1u, w, 5);
          epi_parity ^= 1u << b;
          epi_pending &= ~(1u << b);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          write_box_row<EPI>(smem + (sbuf - sbase) + lane * 128, lane, r0, r1, p.scale);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            store_box(sbuf, col0, row0, l);
            ptx::bulk_commit_group();
          }
        }
      } else if constexpr (EPI == Epilogue::kStoreF32) {
        // FP32 partials (split-K): 32-column boxes of 32 rows x 128 bytes.
#pragma unroll 1
        for (int c = 0; c < Cfg::EPI_COLS / 32; ++c, ++chunk_ctr) {
          const int b = int(chunk_ctr % Cfg::EPI_BUFS);
          const uint32_t sbuf = buf0 + b * Cfg::EPI_BOX_BYTES;
          const int col0 = nb * BN + col_base + c * 32;
          const bool live = rows_live && col0 < p.N;
          if (lane == 0) ptx::bulk_wait_group_read<Cfg::EPI_BUFS - 1>();
          __syncwarp();
          uint32_t r0[32];
          ptx::tmem_ld_32x32b_x32(tacc + uint32_t(c * 32), r0);
          ptx::tmem_ld_wait_regs(r0);
          if (c == Cfg::EPI_COLS / 32 - 1) release_acc(acc);
          if (!live) continue;
          write_box_row_f32(smem + (sbuf - sbase) + lane * 128, lane, r0);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            store_box(sbuf, col0, row0, l);
            ptx::bulk_commit_group();
          }
        }
      } else if constexpr (kDirectStore) {
        // 64 columns per chunk: each lane converts its row and writes eight
        // 16-byte pieces straight to global memory (N % 8 == 0, so a piece
        // is either wholly inside the matrix or wholly outside).
        const int grow = row0 + lane;
#pragma unroll 1
        for (int c = 0; c < Cfg::EPI_COLS / 64; ++c) {
          const int col0 = nb * BN + col_base + c * 64;
          uint32_t r0[32], r1[32];
          const uint32_t taddr = tacc + uint32_t(c * 64);
          ptx::tmem_ld_32x32b_x32(taddr, r0);
          ptx::tmem_ld_32x32b_x32(taddr + 32, r1);
          ptx::tmem_ld_wait_regs(r0);
          ptx::tmem_ld_wait_regs(r1);
          if (c == Cfg::EPI_COLS / 64 - 1) release_acc(acc);
          if (grow >= p.M || col0 >= p.N) continue;
          uint16_t* dst = static_cast<uint16_t*>(p.c_ptr) +
                          (size_t(l) * p.M + size_t(grow)) * size_t(p.N) + col0;
          if ((p.N & 7) == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (col0 + 8 * j >= p.N) break;
              const uint32_t* v = (j < 4) ? &r0[8 * j] : &r1[8 * (j - 4)];
              const uint4 o = epi_chunk<EPI>(v, make_uint4(0, 0, 0, 0), p.scale);
              *reinterpret_cast<uint4*>(dst + 8 * j) = o;
            }
          } else {
            // N not a multiple of 8 (rows are not 16-byte aligned): 2-byte
            // stores, none past column N-1
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint32_t* v = (j < 4) ? &r0[8 * j] : &r1[8 * (j - 4)];
              const uint4 o = epi_chunk<EPI>(v, make_uint4(0, 0, 0, 0), p.scale);
              const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (col0 + 8 * j + e < p.N)
                  dst[8 * j + e] = uint16_t(ow[e >> 1] >> (16 * (e & 1)));
            }
          }
        }
      } else if constexpr (Cfg::EPI_BOX_ROWS < 32) {
        // Boxes of EPI_BOX_ROWS rows: per 64 columns, the warp's 32 rows go
        // out as 32 / EPI_BOX_ROWS boxes, each written by its lanes and
        // stored by TMA (boxes that start past row M are skipped; the map
        // clips the rest).
        static_assert(EPI == Epilogue::kScaleBF16 || EPI == Epilogue::kStoreBF16,
                      "short boxes: plain 16-bit outputs");
        constexpr int HB = 32 / Cfg::EPI_BOX_ROWS;
#pragma unroll 1
        for (int c = 0; c < Cfg::EPI_COLS / 64; ++c) {
          const int col0 = nb * BN + col_base + c * 64;
          uint32_t r0[32], r1[32];
          const uint32_t taddr = tacc + uint32_t(c * 64);
          ptx::tmem_ld_32x32b_x32(taddr, r0);
          ptx::tmem_ld_32x32b_x32(taddr + 32, r1);
          ptx::tmem_ld_wait_regs(r0);
          ptx::tmem_ld_wait_regs(r1);
          if (c == Cfg::EPI_COLS / 64 - 1) release_acc(acc);
          if (!(rows_live && col0 < p.N)) continue;
#pragma unroll 1
          for (int h = 0; h < HB; ++h) {
            if (row0 + h * Cfg::EPI_BOX_ROWS >= p.M) break;  // warp-uniform
            const uint32_t sbuf = buf0 + int(chunk_ctr % Cfg::EPI_BUFS) * Cfg::EPI_BOX_BYTES;
            ++chunk_ctr;
            // The TMA store that last read this buffer must be done with it.
            if (lane == 0) ptx::bulk_wait_group_read<Cfg::EPI_BUFS - 1>();
            __syncwarp();
            if (lane / Cfg::EPI_BOX_ROWS == h)
              write_box_row<EPI>(smem + (sbuf - sbase) + (lane % Cfg::EPI_BOX_ROWS) * 128, lane,
                                 r0, r1, p.scale);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              store_box(sbuf, col0, row0 + h * Cfg::EPI_BOX_ROWS, l);
              ptx::bulk_commit_group();
            }
          }
        }
      } else {
        // The CTA's last whole tile: its MMAs, and so every use of the
        // stages, are complete, so (where they fit) each output box takes a
        // place of its own in the stage memory and the stores go out
        // without waiting for a buffer to be read.
        constexpr bool kLastInStages =
            EPI != Epilogue::kScaledAccBF16 &&
            Cfg::EPI_WARPS * (Cfg::EPI_COLS / 64) * Cfg::EPI_BOX_BYTES <=
                Cfg::STAGES * Cfg::STAGE_BYTES;
        bool last_tile = false;
        if constexpr (kLastInStages) {
          Seg nx;
          last_tile = sg.slot < 0 && !seg_at<Cfg>(p, cluster_id, num_clusters, idx + 1, nx);
        }
#pragma unroll 1
        for (int c = 0; c < Cfg::EPI_COLS / 64; ++c, ++chunk_ctr) {
          const int b = int(chunk_ctr % Cfg::EPI_BUFS);
          const uint32_t sbuf =
              last_tile ? sbase + uint32_t(e * (Cfg::EPI_COLS / 64) + c) * Cfg::EPI_BOX_BYTES
                        : buf0 + b * Cfg::EPI_BOX_BYTES;
          const int col0 = nb * BN + col_base + c * 64;
          const bool live = rows_live && col0 < p.N;
          // The TMA store that last read this buffer must be done with it.
          if (!last_tile) {
            if (lane == 0) ptx::bulk_wait_group_read<Cfg::EPI_BUFS - 1>();
            __syncwarp();
          }
          if constexpr (EPI == Epilogue::kScaledAccBF16) {
            if (live && lane == 0) {
              ptx::mbar_arrive_expect_tx(epi_bar(e, b), Cfg::EPI_BOX_BYTES);
              ptx::tma_load_3d(sbuf, &tmap_c, epi_bar(e, b), col0, row0, l);
            }
            if (live) epi_pending |= 1u << b;
          }
          uint32_t r0[32], r1[32];
          const uint32_t taddr = tacc + uint32_t(c * 64);
          ptx::tmem_ld_32x32b_x32(taddr, r0);
          ptx::tmem_ld_32x32b_x32(taddr + 32, r1);
          ptx::tmem_ld_wait_regs(r0);
          ptx::tmem_ld_wait_regs(r1);
          if (c == Cfg::EPI_COLS / 64 - 1) release_acc(acc);
          if (!live) continue;
          if constexpr (EPI == Epilogue::kStoreBF16 && !kFP4) {
            if (sg.slot >= 0) {
              // stream-K partial tile: two 32-column FP32 boxes into this
              // cluster's workspace slot [cluster*2 + slot][TILE_M][BN] (its
              // map takes the A-scale-factor map's place); the second box
              // takes the next output buffer
              const int sx = col_base + c * 64, sy = int(peer) * Cfg::BM + q * 32;
              const int sz = int(cluster_id) * 2 + sg.slot;
              write_box_row_f32(smem + (sbuf - sbase) + lane * 128, lane, r0);
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                ptx::tma_store_3d(&tmap_sfa, sbuf, sx, sy, sz);
                ptx::bulk_commit_group();
              }
              ++chunk_ctr;
              const uint32_t sbuf2 = buf0 + int(chunk_ctr % Cfg::EPI_BUFS) * Cfg::EPI_BOX_BYTES;
              if (lane == 0) ptx::bulk_wait_group_read<Cfg::EPI_BUFS - 1>();
              __syncwarp();
              write_box_row_f32(smem + (sbuf2 - sbase) + lane * 128, lane, r1);
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                ptx::tma_store_3d(&tmap_sfa, sbuf2, sx + 32, sy, sz);
                ptx::bulk_commit_group();
              }
              continue;
            }
          }
          if constexpr (EPI == Epilogue::kScaledAccBF16) {
            const bool got = wait_bar(epi_bar(e, b), (epi_parity >> b) & 1u, w, 5);
            epi_parity ^= 1u << b;
            epi_pending &= ~(1u << b);
            if (!__all_sync(0xffffffffu, got)) {
              ok = false;
              break;
            }
          }
          write_box_row<EPI>(smem + (sbuf - sbase) + lane * 128, lane, r0, r1, p.scale);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            store_box(sbuf, col0, row0, l);
            ptx::bulk_commit_group();
          }
        }
      }
    }
    if (lane == 0) {
      // Loads that were issued but never waited for (abort path) must land.
      for (int b = 0; b < Cfg::EPI_BUFS; ++b)
        if (epi_pending & (1u << b)) drain_bar(epi_bar(e, b), (epi_parity >> b) & 1u, w);
      // The stores must have read their boxes before the shared memory is
      // released; their writes complete with the grid (a dependent launch
      // sees them after its griddepcontrol.wait), so the CTA does not wait
      // for them.
      ptx::bulk_wait_group_read<0>();
    }
    __syncwarp();
  }

  ptx::tc_fence_before();
  if constexpr (Cfg::CLUSTER > 1) ptx::cluster_sync(); else __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<CG>(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace gb300
