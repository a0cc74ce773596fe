// bf16_scaled_add: out[i] = bf16(float(out[i]) + scale * float(d[i])), the
// second kernel of the unfused LoRA pair ("gemm_dense.rs",
// dense_gemm_tc_scaled_acc doc comment).  HBM-bound streaming kernel: 16-byte
// vector loads/stores, grid sized to a multiple of the SM count.
#include <algorithm>

#include "epilogue_math.cuh"
#include "internal.h"

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

}  // namespace

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
