"""GB300 (sm_103a) dense NT GEMM library: BF16 GEMM, fused LoRA scaled-acc,
ordered FP32 router GEMM and NVFP4 block-scaled GEMM behind a C ABI
(include/gb300gemm.h).  The functions below are the thin torch binding; the
shared library is loaded on first call and must have been built (build.py)."""
from .binding import (  # noqa: F401
    GemmError,
    bf16_scaled_add,
    gemm_bf16_nn,
    gemm_bf16_nt,
    gemm_bf16_nt_ordered,
    gemm_bf16_nt_scaled_acc,
    gemm_bf16_nt_splitk,
    gemm_bf16_nt_splitk_workspace_bytes,
    gemm_bf16_nt_streamk,
    gemm_bf16_nt_streamk_workspace_bytes,
    gemm_nvfp4_bs_splitk,
    gemm_nvfp4_bs_splitk_workspace_bytes,
    gemm_get_device_status,
    gemm_nvfp4_bs,
    gemm_selftest_wait_timeout,
    gemm_testing_set_overrides,
    gemm_w4a16,
    gemm_w4a16_t,
    gemm_w4a16_ws,
    gemm_w4a16_ws_workspace_bytes,
    library_path,
    load,
    status_string,
)
