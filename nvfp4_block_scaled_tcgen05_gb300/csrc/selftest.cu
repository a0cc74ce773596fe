// Failure-path self test: one CTA waits on an mbarrier that nothing arrives
// on, through the same bounded wait the GEMM kernels use.  The wait gives up
// after the requested limit, records a code in the status word and the
// kernel returns normally, leaving the context usable.
#include "internal.h"
#include "watchdog.cuh"

namespace gb300 {

namespace {

__global__ void selftest_timeout_kernel(unsigned int* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);  // expects one arrival that never comes
    abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Watch w{&abort_flag, status, timeout_ns};
    (void)wait_bar(b, 0, w, 0x7F);
  }
}

}  // namespace

int launch_selftest_timeout(int timeout_ms, const DeviceInfo& dev, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(dev.status,
                                                 static_cast<unsigned long long>(timeout_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

}  // namespace gb300
