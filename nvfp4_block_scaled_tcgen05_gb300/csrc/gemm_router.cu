// Order-preserving FP32 "router" GEMM on CUDA cores ("gemm_dense.rs",
// dense_gemm_router / dense_gemm): every output is
//     acc = +0; for k = 0..K-1: acc = fadd_rn(acc, fmul_rn(a[m,k], b[n,k]))
// so the result is bit-identical to the strict sequential loop.  Tensor
// cores reassociate the K sum and are not used here.
//
// Register blocking: each thread owns a TM x TN = 8 x 4 block of outputs
// (32 independent add chains); BK-deep slices of A and B are widened to
// FP32 once and staged k-major in shared memory (double-buffered), so the
// inner loop is two 16-byte loads of A, one of B and 32 multiply/add pairs.
// 64 x 64 block tiles with 16-deep slices (284 blocks of 4 warps for the
// 4510 x 256 router) measured fastest among block tiles of 16-128 rows,
// 32-128 columns, slices of 8-64 and register tiles of 4x4 to 8x8:
// 188 us against 211 us for 32 x 64 blocks of 4 x 4 with 32-deep slices.
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
  auto sstore = [&](int buf) {
#pragma unroll
    for (int i = 0; i < A_PER_T; ++i) {
      const int id = tid + i * kThreads;
      const int row = id % kBM, ch = id / kBM;
      float f[8];
      widen8(ra[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sA[buf][ch * 8 + e][row] = f[e];
    }
#pragma unroll
    for (int i = 0; i < B_PER_T; ++i) {
      const int id = tid + i * kThreads;
      const int row = id % kBN, ch = id / kBN;
      float f[8];
      widen8(rb[i], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) sB[buf][ch * 8 + e][row] = f[e];
    }
  };

  float acc[kTM][kTN];
#pragma unroll
  for (int i = 0; i < kTM; ++i)
#pragma unroll
    for (int j = 0; j < kTN; ++j) acc[i][j] = 0.0f;

  static_assert(kTM == 8 && kTN == 4, "two float4 of A and one of B per k");
  auto step = [&](int buf, int kk) {
    const float4 a0 = *reinterpret_cast<const float4*>(&sA[buf][kk][ty * kTM]);
    const float4 a1 = *reinterpret_cast<const float4*>(&sA[buf][kk][ty * kTM + 4]);
    const float4 b0 = *reinterpret_cast<const float4*>(&sB[buf][kk][tx * kTN]);
    const float a[kTM] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float b[kTN] = {b0.x, b0.y, b0.z, b0.w};
#pragma unroll
    for (int i = 0; i < kTM; ++i)
#pragma unroll
      for (int j = 0; j < kTN; ++j) acc[i][j] = __fadd_rn(acc[i][j], __fmul_rn(a[i], b[j]));
  };

  const int nkb = (K + kBK - 1) / kBK;
  gload(0);
  sstore(0);
  __syncthreads();
  for (int kb = 0; kb < nkb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < nkb) gload((kb + 1) * kBK);
    const int kmax = min(kBK, K - kb * kBK);
    if (kmax == kBK) {
#pragma unroll
      for (int kk = 0; kk < kBK; ++kk) step(buf, kk);
    } else {
#pragma unroll 1
      for (int kk = 0; kk < kmax; ++kk) step(buf, kk);
    }
    if (kb + 1 < nkb) sstore(buf ^ 1);
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < kTM; ++i) {
    const int gm = m0 + ty * kTM + i;
    if (gm >= M) continue;
    const int gn = n0 + tx * kTN;
    float* dst = C + size_t(gm) * N + gn;
    if (gn + kTN <= N && (N % 4) == 0) {
      *reinterpret_cast<float4*>(dst) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    } else {
#pragma unroll
      for (int j = 0; j < kTN; ++j)
        if (gn + j < N) dst[j] = acc[i][j];
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
