"""The allocation-free split-K entry point (gemm_bf16_nt_splitk_static).

It serves callers that cannot allocate device memory themselves (a host
framework that owns the whole device pool, a serving loop that must not call
the CUDA allocator after warm-up, a plugin handed raw pointers but no
allocator).  Its workspace is a fixed scratch array inside the library, so
this test calls it straight through the C ABI, twice in a row on one stream
with different inputs, and checks each result against the workspace-taking
entry point, with the tolerance the other parity tests use.  It lives in a
file of its own that pytest collects last."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import bf16_val, bits16, check_close16, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_tcgen05_gb300 import binding
    so = ctypes.CDLL(binding.library_path())
    f = so.gemm_bf16_nt_splitk_static
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    return so


def amax(x):
    return float(np.abs(bf16_val(x)).max())


def test_static_scratch_splitk_twice_matches_workspace_variant(lib):
    import nvfp4_block_scaled_tcgen05_gb300 as g
    M, N, K, splits = 640, 512, 1032, 3
    A = synth.bf16_normal((M, K), 1.0, 201)
    B1 = synth.bf16_normal((N, K), 1.0, 202)
    B2 = synth.bf16_normal((N, K), 0.5, 203)
    Ad, B1d, B2d = to_dev_bf16(A), to_dev_bf16(B1), to_dev_bf16(B2)
    C1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    C2 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row, no synchronisation between them
    assert lib.gemm_bf16_nt_splitk_static(Ad.data_ptr(), B1d.data_ptr(), C1.data_ptr(),
                                          M, N, K, splits, stream) == 0
    assert lib.gemm_bf16_nt_splitk_static(Ad.data_ptr(), B2d.data_ptr(), C2.data_ptr(),
                                          M, N, K, splits, stream) == 0
    torch.cuda.synchronize()
    assert g.gemm_get_device_status() == 0
    for C, Bh, Bd, name in ((C1, B1, B1d, "first call"), (C2, B2, B2d, "second call")):
        ref = bits16(g.gemm_bf16_nt_splitk(Ad, Bd, splits))
        check_close16(bits16(C), ref, K, amax(A), amax(Bh), what=f"static scratch, {name}")
    # and against the oracle, for the second call
    rows = np.arange(0, M, 37)
    check_close16(bits16(C2)[rows], oracle.gemm_bf16_nt(A, B2, rows=rows), K, amax(A), amax(B2),
                  what="static scratch vs oracle")


def test_static_scratch_rejects_problems_over_the_limit(lib):
    # 4 splits of 4096 x 4096 FP32 partials = 256 MiB > the 32 MiB scratch
    P = 0x10000
    assert lib.gemm_bf16_nt_splitk_static(P, 2 * P, 3 * P, 4096, 4096, 4096, 4, None) == 2
