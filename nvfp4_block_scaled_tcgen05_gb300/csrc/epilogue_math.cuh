// Element arithmetic shared by the GEMM epilogues and the standalone
// bf16_scaled_add kernel.  Keeping one definition is what makes the fused
// scaled-acc epilogue bit-identical to "GEMM into a BF16 scratch, then
// bf16_scaled_add" ("gemm_dense.rs", dense_gemm_tc_scaled_acc).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gb300 {

// Two FP32 values (given as bit patterns) -> bf16x2, round to nearest even;
// the first value goes to the low half (lower address).
__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(uint32_t lo, uint32_t hi) {
  __half2 h = __floats2half2_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// out = bf16( float(out) + scale * float(d) ), the product and the sum each
// rounded to FP32 separately (never fused), applied to a bf16 pair.
__device__ __forceinline__ uint32_t scaled_acc_bf16x2(uint32_t out2, uint32_t d2, float scale) {
  const float r0 = __fadd_rn(bf16_lo(out2), __fmul_rn(scale, bf16_lo(d2)));
  const float r1 = __fadd_rn(bf16_hi(out2), __fmul_rn(scale, bf16_hi(d2)));
  return pack_bf16x2(__float_as_uint(r0), __float_as_uint(r1));
}

}  // namespace gb300
