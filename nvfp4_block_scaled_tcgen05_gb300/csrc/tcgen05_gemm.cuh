// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   C[l][m][n] = epilogue( sum_k A[l][m][k] * B[l][n][k] )      (NT layout)
//
// Operands: BF16 (kind::f16) or packed e2m1 with e4m3 block scales
// (kind::mxf4nvf4, scale_vec::4X).  One CTA per SM walks the output tiles
// tile = blockIdx.x + i*gridDim.x in grouped-M raster order.  Roles:
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) and, for NVFP4,
//               the 512-byte scale atoms, into a STAGES-deep smem ring;
//   warp 1      allocates TMEM; lane 0 issues tcgen05.mma into a TMEM
//               accumulator (two when the column budget allows) and, for
//               NVFP4, tcgen05.cp's the scale atoms into TMEM first;
//   warps 2..5  epilogue: tcgen05.ld -> convert (bf16 / fp16 / scaled-acc)
//               -> swizzled smem box -> TMA store; for scaled-acc the old
//               output box is TMA-loaded into the same smem first.
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

namespace gb300 {

enum class Operand : int { kBF16 = 0, kNVFP4 = 1 };
enum class Epilogue : int { kStoreBF16 = 0, kScaledAccBF16 = 1, kStoreFP16 = 2 };

struct GemmParams {
  int M, N, K, L;                 // K in elements
  int num_m_blocks, num_n_blocks, num_k_blocks, total_tiles;
  int rest_m, rest_n, rest_k;     // NVFP4 scale layout extents: M/128, N/128, K/64
  float scale;                    // scaled-acc factor
  const uint8_t* sfa;             // NVFP4 scale buffers (hardware layout)
  const uint8_t* sfb;
  unsigned int* status;           // device status word
  unsigned long long timeout_ns;  // bound on every wait
};

template <Operand OP, int BN_, int STAGES_>
struct TileCfg {
  static constexpr Operand kOp = OP;
  static constexpr bool kFP4 = (OP == Operand::kNVFP4);
  static constexpr int BM = 128;
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static constexpr int BK = kFP4 ? 256 : 64;        // K elements per stage = 128 bytes per row
  static constexpr int KX = kFP4 ? 128 : 64;        // TMA x-extent per stage (bytes or elements)
  static constexpr int MMA_K = kFP4 ? 64 : 16;      // K per MMA = 32 bytes per row
  static constexpr int KSTEPS = BK / MMA_K;         // 4 MMAs per stage
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int SF_ATOM = 512;               // 128 rows x 4 scales
  static constexpr int SFB_ATOMS_N = kFP4 ? BN / 128 : 0;
  static constexpr int SFA_BYTES = kFP4 ? KSTEPS * SF_ATOM : 0;
  static constexpr int SFB_BYTES = kFP4 ? SFB_ATOMS_N * KSTEPS * SF_ATOM : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int EPI_BOX_BYTES = 32 * 128;    // 32 rows x 64 16-bit values
  static constexpr int EPI_BUFS = 2;
  static constexpr int EPI_BYTES = 4 * EPI_BUFS * EPI_BOX_BYTES;
  // TMEM columns: accumulators first, then one scale slot per smem stage.
  static constexpr int SF_COLS = kFP4 ? KSTEPS * 4 * (1 + SFB_ATOMS_N) : 0;
  static constexpr int NUM_ACC = (2 * BN + STAGES * SF_COLS <= 512) ? 2 : 1;
  static constexpr int SF_TMEM_BASE = NUM_ACC * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(NUM_ACC * BN + STAGES * SF_COLS <= TMEM_COLS, "TMEM column budget");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(!kFP4 || BN % 128 == 0, "NVFP4 BN must cover whole 128-row scale atoms");
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2], epi[4][2], mma_done
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 8 + 1;
  static constexpr int BAR_BYTES = NUM_BARS * 8 + 16;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget (227 KB per CTA)");
  static constexpr int THREADS = 192;
  static constexpr int GROUP_M = 8;

  // Instruction descriptor.  kind::f16: D=F32 (bits 4-5 = 1), A=B=BF16
  // (bits 7-9 = 1, 10-12 = 1), both K-major, N>>3 in bits 17-22, M>>4 in
  // bits 24-28.  kind::mxf4nvf4: A=B=E2M1 (1), scale type UE4M3 (bit 23 = 0),
  // scale ids 0, dense K=64.
  __host__ __device__ static constexpr uint32_t idesc() {
    return kFP4 ? ((1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24))
                : ((1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
                   (uint32_t(BM >> 4) << 24));
  }
};

// Watchdog state shared by the roles of one CTA.
struct Watch {
  volatile uint32_t* abort;
  unsigned int* status;
  unsigned long long timeout_ns;
};

// Bounded wait on an mbarrier phase.  Returns false if the CTA aborted or
// this wait ran out (then it records `code` and raises the abort flag).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Watch& w,
                                         uint32_t code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (ptx::globaltimer() - t0 > w.timeout_ns) {
      *w.abort = 1u;
      atomicCAS(w.status, 0u, 0x100u | code);
      return false;
    }
  }
}

// Bounded wait used while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, const Watch& w) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > w.timeout_ns) {
      atomicCAS(w.status, 0u, 0x1FFu);
      return;
    }
  }
}

template <class Cfg>
__device__ __forceinline__ void decode_tile(int tile, const GemmParams& p, int& l, int& mb,
                                            int& nb) {
  const int per_batch = p.num_m_blocks * p.num_n_blocks;
  l = tile / per_batch;
  const int t = tile - l * per_batch;
  const int group_tiles = Cfg::GROUP_M * p.num_n_blocks;
  const int g = t / group_tiles;
  const int first_m = g * Cfg::GROUP_M;
  const int gm = min(p.num_m_blocks - first_m, Cfg::GROUP_M);
  const int r = t - g * group_tiles;
  mb = first_m + r % gm;
  nb = r / gm;
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

template <class Cfg, Epilogue EPI>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tcgen05_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_c, const GemmParams p) {
  constexpr int STAGES = Cfg::STAGES;
  constexpr int BN = Cfg::BN;
  constexpr bool kFP4 = Cfg::kFP4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t epi_base = sbase + STAGES * Cfg::STAGE_BYTES;
  const uint32_t bar_base = epi_base + Cfg::EPI_BYTES;
  auto stage_a = [&](int s) { return sbase + s * Cfg::STAGE_BYTES; };
  auto stage_b = [&](int s) { return sbase + s * Cfg::STAGE_BYTES + Cfg::A_BYTES; };
  auto stage_sfa = [&](int s) { return stage_b(s) + Cfg::B_BYTES; };
  auto stage_sfb = [&](int s) { return stage_sfa(s) + Cfg::SFA_BYTES; };
  auto full_bar = [&](int s) { return bar_base + 8 * s; };
  auto empty_bar = [&](int s) { return bar_base + 8 * (STAGES + s); };
  auto acc_full = [&](int b) { return bar_base + 8 * (2 * STAGES + b); };
  auto acc_empty = [&](int b) { return bar_base + 8 * (2 * STAGES + 2 + b); };
  auto epi_bar = [&](int q, int b) { return bar_base + 8 * (2 * STAGES + 4 + 2 * q + b); };
  const uint32_t mma_done = bar_base + 8 * (2 * STAGES + 12);
  uint8_t* misc = smem + (bar_base - sbase) + 8 * Cfg::NUM_BARS;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(misc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(misc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(acc_full(b), 1);
      ptx::mbar_init(acc_empty(b), 4);
    }
    for (int q = 0; q < 4; ++q)
      for (int b = 0; b < 2; ++b) ptx::mbar_init(epi_bar(q, b), 1);
    ptx::mbar_init(mma_done, 1);
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_a);
    ptx::prefetch_tmap(&tmap_b);
    ptx::prefetch_tmap(&tmap_c);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(tmem_slot)), Cfg::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const Watch w{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;  // bit s: stage s has a load in flight / its parity
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x) {
        int l, mb, nb;
        decode_tile<Cfg>(tile, p, l, mb, nb);
        int sfb_atoms = 0;
        if constexpr (kFP4) sfb_atoms = min(Cfg::SFB_ATOMS_N, p.rest_n - nb * Cfg::SFB_ATOMS_N);
        const uint32_t tx = Cfg::A_BYTES + Cfg::B_BYTES + Cfg::SFA_BYTES +
                            uint32_t(sfb_atoms) * Cfg::KSTEPS * Cfg::SF_ATOM;
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!wait_bar(empty_bar(stage), phase ^ 1u, w, 1)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(full_bar(stage), tx);
          ptx::tma_load_3d(stage_a(stage), &tmap_a, full_bar(stage), kb * Cfg::KX, mb * Cfg::BM, l);
          ptx::tma_load_3d(stage_b(stage), &tmap_b, full_bar(stage), kb * Cfg::KX, nb * BN, l);
          if constexpr (kFP4) {
            // 4 consecutive atoms (tile_k = 4kb .. 4kb+3) are contiguous: 2 KB per 128 rows.
            const size_t a_off =
                (size_t(size_t(l) * p.rest_m + mb) * p.rest_k + size_t(4 * kb)) * Cfg::SF_ATOM;
            ptx::bulk_load(stage_sfa(stage), p.sfa + a_off, Cfg::KSTEPS * Cfg::SF_ATOM,
                           full_bar(stage));
            for (int at = 0; at < sfb_atoms; ++at) {
              const size_t b_off = (size_t(size_t(l) * p.rest_n + nb * Cfg::SFB_ATOMS_N + at) *
                                        p.rest_k +
                                    size_t(4 * kb)) *
                                   Cfg::SF_ATOM;
              ptx::bulk_load(stage_sfb(stage) + at * Cfg::KSTEPS * Cfg::SF_ATOM, p.sfb + b_off,
                             Cfg::KSTEPS * Cfg::SF_ATOM, full_bar(stage));
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
      // Every load issued must have landed before the CTA may exit.
      for (int s = 0; s < STAGES; ++s)
        if (armed & (1u << s)) drain_bar(full_bar(s), (armed_parity >> s) & 1u, w);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = Cfg::idesc();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x, ++it) {
        const int acc = it % Cfg::NUM_ACC;
        const uint32_t acc_phase = uint32_t(it / Cfg::NUM_ACC) & 1u;
        if (!wait_bar(acc_empty(acc), acc_phase ^ 1u, w, 2)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!wait_bar(full_bar(stage), phase, w, 3)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = stage_a(stage), b0 = stage_b(stage);
          if constexpr (kFP4) {
            const uint32_t sfa_t = tmem_base + uint32_t(Cfg::SF_TMEM_BASE + stage * Cfg::SF_COLS);
            const uint32_t sfb_t = sfa_t + Cfg::KSTEPS * 4;
#pragma unroll
            for (int j = 0; j < Cfg::KSTEPS; ++j) {
              ptx::tc_cp_32x128b_warpx4(sfa_t + 4 * j,
                                        ptx::smem_desc(stage_sfa(stage) + j * Cfg::SF_ATOM, 0, 128, 0));
#pragma unroll
              for (int at = 0; at < Cfg::SFB_ATOMS_N; ++at)
                ptx::tc_cp_32x128b_warpx4(
                    sfb_t + j * 4 * Cfg::SFB_ATOMS_N + 4 * at,
                    ptx::smem_desc(stage_sfb(stage) + (at * Cfg::KSTEPS + j) * Cfg::SF_ATOM, 0, 128,
                                   0));
            }
#pragma unroll
            for (int j = 0; j < Cfg::KSTEPS; ++j)
              ptx::mma_nvf4(d_tmem, ptx::sw128_kmajor_desc(a0 + 32 * j),
                            ptx::sw128_kmajor_desc(b0 + 32 * j), idesc, sfa_t + 4 * j,
                            sfb_t + j * 4 * Cfg::SFB_ATOMS_N, (kb | j) != 0);
          } else {
            // K tail: the zero-filled part of the last stage needs no MMA.
            const int krem = p.K - kb * Cfg::BK;
            const int nsteps = krem >= Cfg::BK ? Cfg::KSTEPS : (krem + Cfg::MMA_K - 1) / Cfg::MMA_K;
#pragma unroll
            for (int j = 0; j < Cfg::KSTEPS; ++j)
              if (j < nsteps)
                ptx::mma_bf16(d_tmem, ptx::sw128_kmajor_desc(a0 + 32 * j),
                              ptx::sw128_kmajor_desc(b0 + 32 * j), idesc, (kb | j) != 0);
          }
          ptx::tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit(acc_full(acc));
      }
      // Every MMA / copy issued must be complete before TMEM is released.
      ptx::tc_commit(mma_done);
      drain_bar(mma_done, 0, w);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const uint32_t lane_off = uint32_t(q * 32) << 16;
    const uint32_t buf0 = epi_base + q * Cfg::EPI_BUFS * Cfg::EPI_BOX_BYTES;
    uint32_t chunk_ctr = 0;
    uint32_t epi_parity = 0;     // bit b: parity of the next wait on epi_bar(q, b)
    uint32_t epi_pending = 0;    // bit b: a load into buffer b has not been waited for
    bool ok = true;
    int it = 0;
    for (int tile = blockIdx.x; ok && tile < p.total_tiles; tile += gridDim.x, ++it) {
      int l, mb, nb;
      decode_tile<Cfg>(tile, p, l, mb, nb);
      const int acc = it % Cfg::NUM_ACC;
      const uint32_t acc_phase = uint32_t(it / Cfg::NUM_ACC) & 1u;
      ok = __all_sync(0xffffffffu, wait_bar(acc_full(acc), acc_phase, w, 4));
      if (!ok) break;
      ptx::tc_fence_after();
      const int row0 = mb * Cfg::BM + q * 32;
      const bool rows_live = row0 < p.M;
#pragma unroll 1
      for (int c = 0; c < BN / 64; ++c, ++chunk_ctr) {
        const int b = int(chunk_ctr & 1u);
        const uint32_t sbuf = buf0 + b * Cfg::EPI_BOX_BYTES;
        const int col0 = nb * BN + c * 64;
        const bool live = rows_live && col0 < p.N;
        // The TMA store that last read this buffer must be done with it.
        if (lane == 0) ptx::bulk_wait_group_read<1>();
        __syncwarp();
        if constexpr (EPI == Epilogue::kScaledAccBF16) {
          if (live && lane == 0) {
            ptx::mbar_arrive_expect_tx(epi_bar(q, b), Cfg::EPI_BOX_BYTES);
            ptx::tma_load_3d(sbuf, &tmap_c, epi_bar(q, b), col0, row0, l);
          }
          if (live) epi_pending |= 1u << b;
        }
        uint32_t r0[32], r1[32];
        const uint32_t taddr = tmem_base + lane_off + uint32_t(acc * BN + c * 64);
        ptx::tmem_ld_32x32b_x32(taddr, r0);
        ptx::tmem_ld_32x32b_x32(taddr + 32, r1);
        ptx::tmem_ld_wait_regs(r0);
        ptx::tmem_ld_wait_regs(r1);
        if (c == BN / 64 - 1) {
          // Accumulator fully read: hand it back to the MMA warp.
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(acc_empty(acc));
        }
        if (!live) continue;
        if constexpr (EPI == Epilogue::kScaledAccBF16) {
          const bool got = wait_bar(epi_bar(q, b), (epi_parity >> b) & 1u, w, 5);
          epi_parity ^= 1u << b;
          epi_pending &= ~(1u << b);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
        }
        uint8_t* row = smem + (sbuf - sbase) + lane * 128;
        const float scale = p.scale;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4* chunk = reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4));
          uint4 old = make_uint4(0, 0, 0, 0);
          if constexpr (EPI == Epilogue::kScaledAccBF16) old = *chunk;
          *chunk = epi_chunk<EPI>(&r0[8 * j], old, scale);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4* chunk = reinterpret_cast<uint4*>(row + (((j + 4) ^ (lane & 7)) << 4));
          uint4 old = make_uint4(0, 0, 0, 0);
          if constexpr (EPI == Epilogue::kScaledAccBF16) old = *chunk;
          *chunk = epi_chunk<EPI>(&r1[8 * j], old, scale);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_3d(&tmap_c, sbuf, col0, row0, l);
          ptx::bulk_commit_group();
        }
      }
    }
    if (lane == 0) {
      // Loads that were issued but never waited for (abort path) must land.
      for (int b = 0; b < 2; ++b)
        if (epi_pending & (1u << b)) drain_bar(epi_bar(q, b), (epi_parity >> b) & 1u, w);
      ptx::bulk_wait_group<0>();
    }
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace gb300
