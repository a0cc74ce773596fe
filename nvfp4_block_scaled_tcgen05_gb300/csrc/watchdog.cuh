// Bounded waits shared by the kernels: every spin on an mbarrier gives up
// after a time limit (%globaltimer), records where in the device status word
// and raises a CTA-wide abort flag, so a broken pipeline returns an error
// instead of hanging the GPU.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace gb300 {

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

__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = ptx::globaltimer();
  while (ptx::globaltimer() - t0 < ns) {
  }
}

}  // namespace gb300
