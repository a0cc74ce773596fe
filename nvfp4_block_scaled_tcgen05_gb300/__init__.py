"""GB300 (sm_103a) dense NT GEMM library: BF16 GEMM, fused LoRA scaled-acc,
ordered FP32 router GEMM and NVFP4 block-scaled GEMM behind a C ABI."""
