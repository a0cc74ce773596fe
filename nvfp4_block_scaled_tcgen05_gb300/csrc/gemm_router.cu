// Order-preserving FP32 "router" GEMM on CUDA cores ("gemm_dense.rs",
// dense_gemm_router / dense_gemm): every output is
//     acc = +0; for k = 0..K-1: acc = fadd_rn(acc, fmul_rn(a[m,k], b[n,k]))
// so the result is bit-identical to the strict sequential loop.  Tensor
// cores reassociate the K sum and are not used here.
//
// Fused multiply-add without changing a bit: a and b are BF16 (8
// significant bits), so a product has at most 16 and is exact in FP32
// whenever it is a normal number; then fma(a, b, acc) = RN(acc + a*b) =
// fadd_rn(acc, fmul_rn(a, b)).  Every nonzero operand in [2^-63, 2^63)
// keeps every product normal (|a*b| in [2^-126, 2^126)); zeros give exact
// zeros, and an accumulator that only ever adds +0 or nonzero values is
// never -0.  So each staged K slice is checked as it is widened: if any A
// or B value of the slice lies outside that range (subnormal, tiny, huge,
// inf or NaN), the block runs that slice with separate multiplies and
// adds; otherwise with packed two-lane fused multiply-adds
// (fma.rn.f32x2 on rows 2i, 2i+1 of one column).  Measured on the 4510 x
// 256 x 2048 router: 131 us against 188 us for the separate scalar
// operations, which were bound by instruction issue (76 % of cycles
// issuing, the FP32 pipe 67 % busy).
//
// Register blocking: each thread owns a TM x TN = 8 x 4 block of outputs
// (32 independent add chains); BK-deep slices of A and B are widened to
// FP32 once and staged k-major in shared memory (double-buffered), so the
// inner loop is two 16-byte loads of A, one of B and 16 packed fused
// multiply-adds (or 32 multiply/add pairs in a checked slice).
// 64 x 64 block tiles with 16-deep slices (284 blocks of 4 warps for the
// 4510 x 256 router) measured fastest among block tiles of 16-128 rows,
// 32-128 columns, slices of 8-64 and register tiles of 4x4 to 8x8, with
// the separate operations and again with the packed ones.
#include <algorithm>

#include "internal.h"

namespace gb300 {

namespace {

constexpr int kBM = 64, kBN = 64, kBK = 16, kTM = 8, kTN = 4;
constexpr int kTX = kBN / kTN;  // 16 threads along n
constexpr int kTY = kBM / kTM;  // 8 threads along m
constexpr int kThreads = kTX * kTY;
constexpr int kPad = 4;
constexpr int kChunks = kBK / 8;  // 16-byte chunks per row per slice

// Any of the 8 BF16 values outside {0} U +-[2^-63, 2^63): biased exponent
// below 64 (subnormal or tiny) or above 189 (huge, inf, NaN).
__device__ __forceinline__ bool outside_exact_range(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  bool r = false;
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t x = (w[q] >> (16 * h)) & 0x7FFFu;
      const uint32_t e = x >> 7;
      r |= (x != 0u) && (e < 64u || e > 189u);
    }
  return r;
}

// Packed FP32 pairs (low lane = first value).
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// d = a * b + d per lane, one rounding (exact products only, see above)
__device__ __forceinline__ void fma2_rn(uint64_t& d, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

__device__ __forceinline__ void widen8(uint4 v, float* f) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16);
  f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16);
  f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

__global__ void __launch_bounds__(kThreads)
    router_kernel(const uint16_t* __restrict__ A, const uint16_t* __restrict__ B,
                  float* __restrict__ C, int M, int N, int K) {
  __shared__ __align__(16) float sA[2][kBK][kBM + kPad];
  __shared__ __align__(16) float sB[2][kBK][kBN + kPad];
  const int tid = threadIdx.x;
  const int tx = tid % kTX, ty = tid / kTX;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;

  constexpr int A_PER_T = kBM * kChunks / kThreads;  // 1
  constexpr int B_PER_T = kBN * kChunks / kThreads;  // 1
  static_assert(A_PER_T * kThreads == kBM * kChunks && B_PER_T * kThreads == kBN * kChunks, "");
  uint4 ra[A_PER_T], rb[B_PER_T];

  // Chunk id -> (row, 16-byte chunk): consecutive threads take consecutive
  // rows of one chunk column, so the transposed shared-memory stores of a
  // warp hit 32 different banks.
  auto gload = [&](int k0) {
#pragma unroll
    for (int i = 0; i < A_PER_T; ++i) {
      const int id = tid + i * kThreads;
      const int row = id % kBM, ch = id / kBM;
      const int gm = m0 + row, gk = k0 + ch * 8;
      ra[i] = (gm < M && gk < K) ? __ldg(reinterpret_cast<const uint4*>(A + size_t(gm) * K + gk))
                                 : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < B_PER_T; ++i) {
      const int id = tid + i * kThreads;
      const int row = id % kBN, ch = id / kBN;
      const int gn = n0 + row, gk = k0 + ch * 8;
      rb[i] = (gn < N && gk < K) ? __ldg(reinterpret_cast<const uint4*>(B + size_t(gn) * K + gk))
                                 : make_uint4(0, 0, 0, 0);
    }
  };
  bool wild = false;  // this thread staged a value outside the exact range
  auto sstore = [&](int buf) {
#pragma unroll
    for (int i = 0; i < A_PER_T; ++i) {
      const int id = tid + i * kThreads;
      const int row = id % kBM, ch = id / kBM;
      float f[8];
      wild |= outside_exact_range(ra[i]);
      widen8(ra[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sA[buf][ch * 8 + e][row] = f[e];
    }
#pragma unroll
    for (int i = 0; i < B_PER_T; ++i) {
      const int id = tid + i * kThreads;
      const int row = id % kBN, ch = id / kBN;
      float f[8];
      wild |= outside_exact_range(rb[i]);
      widen8(rb[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sB[buf][ch * 8 + e][row] = f[e];
    }
  };

  // acc[i][j]: the outputs of rows 2i (low lane) and 2i+1 of column j
  uint64_t acc[kTM / 2][kTN];
#pragma unroll
  for (int i = 0; i < kTM / 2; ++i)
#pragma unroll
    for (int j = 0; j < kTN; ++j) acc[i][j] = 0ull;  // +0, +0

  static_assert(kTM == 8 && kTN == 4, "two float4 of A and one of B per k");
  auto step = [&](int buf, int kk, bool exact_fma) {
    const float4 a0 = *reinterpret_cast<const float4*>(&sA[buf][kk][ty * kTM]);
    const float4 a1 = *reinterpret_cast<const float4*>(&sA[buf][kk][ty * kTM + 4]);
    const float4 b0 = *reinterpret_cast<const float4*>(&sB[buf][kk][tx * kTN]);
    const float a[kTM] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float b[kTN] = {b0.x, b0.y, b0.z, b0.w};
    if (exact_fma) {
#pragma unroll
      for (int j = 0; j < kTN; ++j) {
        const uint64_t bb = pack2(b[j], b[j]);
#pragma unroll
        for (int i = 0; i < kTM / 2; ++i) fma2_rn(acc[i][j], pack2(a[2 * i], a[2 * i + 1]), bb);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kTN; ++j)
#pragma unroll
        for (int i = 0; i < kTM / 2; ++i) {
          float lo, hi;
          unpack2(acc[i][j], lo, hi);
          lo = __fadd_rn(lo, __fmul_rn(a[2 * i], b[j]));
          hi = __fadd_rn(hi, __fmul_rn(a[2 * i + 1], b[j]));
          acc[i][j] = pack2(lo, hi);
        }
    }
  };

  // Slices past K are staged as zeros, whose products (+0) leave the
  // accumulator unchanged, so every slice runs all kBK steps.
  const int nkb = (K + kBK - 1) / kBK;
  gload(0);
  sstore(0);
  bool fma_ok = !__syncthreads_or(wild);
  for (int kb = 0; kb < nkb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < nkb) gload((kb + 1) * kBK);
    if (fma_ok) {
#pragma unroll
      for (int kk = 0; kk < kBK; ++kk) step(buf, kk, true);
    } else {
#pragma unroll 1
      for (int kk = 0; kk < kBK; ++kk) step(buf, kk, false);
    }
    wild = false;
    if (kb + 1 < nkb) sstore(buf ^ 1);
    fma_ok = !__syncthreads_or(wild);
  }

#pragma unroll
  for (int i = 0; i < kTM; ++i) {
    const int gm = m0 + ty * kTM + i;
    if (gm >= M) continue;
    const int gn = n0 + tx * kTN;
    float* dst = C + size_t(gm) * N + gn;
    float r[kTN], other;
#pragma unroll
    for (int j = 0; j < kTN; ++j) {
      if (i & 1) unpack2(acc[i / 2][j], other, r[j]);
      else unpack2(acc[i / 2][j], r[j], other);
    }
    (void)other;
    if (gn + kTN <= N && (N % 4) == 0) {
      *reinterpret_cast<float4*>(dst) = make_float4(r[0], r[1], r[2], r[3]);
    } else {
#pragma unroll
      for (int j = 0; j < kTN; ++j)
        if (gn + j < N) dst[j] = r[j];
    }
  }
}

}  // namespace

int launch_gemm_router(const void* A, const void* B, float* C, int M, int N, int K,
                       const DeviceInfo& dev, cudaStream_t stream) {
  (void)dev;
  const dim3 grid((N + kBN - 1) / kBN, (M + kBM - 1) / kBM);
  router_kernel<<<grid, kThreads, 0, stream>>>(static_cast<const uint16_t*>(A),
                                               static_cast<const uint16_t*>(B), C, M, N, K);
  return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

}  // namespace gb300
