// bf16_scaled_add: out[i] = bf16(float(out[i]) + scale * float(d[i])), the
// second kernel of the unfused LoRA pair ("gemm_dense.rs",
// dense_gemm_tc_scaled_acc doc comment), and the ordered split-K reduce.
// HBM-bound streaming kernels: 16-byte vector loads/stores, grid sized to a
// multiple of the SM count.
#include <algorithm>

#include "epilogue_math.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    scaled_add_kernel(uint16_t* __restrict__ out, const uint16_t* __restrict__ d, float scale,
                      long n) {
  const long nvec = n / 8;
  uint4* o4 = reinterpret_cast<uint4*>(out);
  const uint4* d4 = reinterpret_cast<const uint4*>(d);
  const long stride = long(gridDim.x) * kThreads;
  for (long i = long(blockIdx.x) * kThreads + threadIdx.x; i < nvec; i += stride) {
    uint4 o = o4[i];
    const uint4 v = __ldg(d4 + i);
    o.x = scaled_acc_bf16x2(o.x, v.x, scale);
    o.y = scaled_acc_bf16x2(o.y, v.y, scale);
    o.z = scaled_acc_bf16x2(o.z, v.z, scale);
    o.w = scaled_acc_bf16x2(o.w, v.w, scale);
    o4[i] = o;
  }
  const long tail = n - nvec * 8;
  if (blockIdx.x == 0 && threadIdx.x < tail) {
    const long idx = nvec * 8 + threadIdx.x;
    out[idx] = uint16_t(scaled_acc_bf16x2(out[idx], d[idx], scale) & 0xFFFFu);
  }
}

// C[i] = out16(ws[0][i] + ws[1][i] + ... + ws[S-1][i]), FP32 adds in split
// order (deterministic), then one RNE to BF16 or FP16; 8 outputs per thread,
// 16-byte accesses.
template <bool kF16>
__device__ __forceinline__ uint32_t pack_out16(uint32_t lo, uint32_t hi) {
  if constexpr (kF16) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

template <bool kF16>
__global__ void __launch_bounds__(kThreads)
    splitk_reduce_kernel(const float* __restrict__ ws, uint16_t* __restrict__ C, size_t n,
                         int splits) {
  // launched as a programmatic dependent of the split-K GEMM: wait for its
  // end (and its partials) here, after this grid's launch overlapped it.
  // The next grid on the stream may be scheduled at once (it waits for
  // this one's end before touching memory this one writes).
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  const size_t nvec = n / 8;
  const size_t stride = size_t(gridDim.x) * kThreads;
  for (size_t i = size_t(blockIdx.x) * kThreads + threadIdx.x; i < nvec; i += stride) {
    float4 a = __ldg(reinterpret_cast<const float4*>(ws) + 2 * i);
    float4 b = __ldg(reinterpret_cast<const float4*>(ws) + 2 * i + 1);
    for (int s = 1; s < splits; ++s) {
      const float4* src = reinterpret_cast<const float4*>(ws + size_t(s) * n) + 2 * i;
      const float4 x = __ldg(src), y = __ldg(src + 1);
      a.x = __fadd_rn(a.x, x.x); a.y = __fadd_rn(a.y, x.y);
      a.z = __fadd_rn(a.z, x.z); a.w = __fadd_rn(a.w, x.w);
      b.x = __fadd_rn(b.x, y.x); b.y = __fadd_rn(b.y, y.y);
      b.z = __fadd_rn(b.z, y.z); b.w = __fadd_rn(b.w, y.w);
    }
    uint4 o;
    o.x = pack_out16<kF16>(__float_as_uint(a.x), __float_as_uint(a.y));
    o.y = pack_out16<kF16>(__float_as_uint(a.z), __float_as_uint(a.w));
    o.z = pack_out16<kF16>(__float_as_uint(b.x), __float_as_uint(b.y));
    o.w = pack_out16<kF16>(__float_as_uint(b.z), __float_as_uint(b.w));
    reinterpret_cast<uint4*>(C)[i] = o;
  }
  const size_t tail = n - nvec * 8;
  if (blockIdx.x == 0 && threadIdx.x < tail) {
    const size_t idx = nvec * 8 + threadIdx.x;
    float a = ws[idx];
    for (int s = 1; s < splits; ++s) a = __fadd_rn(a, ws[size_t(s) * n + idx]);
    C[idx] = uint16_t(pack_out16<kF16>(__float_as_uint(a), 0u) & 0xFFFFu);
  }
}

}  // namespace

template <bool kF16>
int launch_reduce(const float* ws, void* C, size_t n, int splits, const DeviceInfo& dev,
                  cudaStream_t stream) {
  const size_t nvec = n / 8;
  const size_t want = (nvec + kThreads - 1) / kThreads;
  const int grid = int(std::max<size_t>(1, std::min<size_t>(want, size_t(dev.num_sms) * 8)));
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  uint16_t* out = static_cast<uint16_t*>(C);
  if (cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<kF16>, ws, out, n, splits) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}

int launch_splitk_reduce(const float* ws, void* C, size_t n, int splits, const DeviceInfo& dev,
                         cudaStream_t stream) {
  return launch_reduce<false>(ws, C, n, splits, dev, stream);
}

int launch_splitk_reduce_f16(const float* ws, void* C, size_t n, int splits, const DeviceInfo& dev,
                             cudaStream_t stream) {
  return launch_reduce<true>(ws, C, n, splits, dev, stream);
}

int launch_scaled_add(void* out, const void* d, float scale, long n, const DeviceInfo& dev,
                      cudaStream_t stream) {
  const long nvec = n / 8;
  const long want = (nvec + kThreads - 1) / kThreads;
  const int grid = int(std::max(1L, std::min(want, long(dev.num_sms) * 8)));
  scaled_add_kernel<<<grid, kThreads, 0, stream>>>(static_cast<uint16_t*>(out),
                                                   static_cast<const uint16_t*>(d), scale, n);
  return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

}  // namespace gb300
