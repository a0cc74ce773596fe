"""The allocation-free split-K entry point (gemm_bf16_nt_splitk_static).

It serves callers that cannot allocate device memory themselves (a host
framework that owns the whole device pool, a serving loop that must not call
the CUDA allocator after warm-up, a plugin handed raw pointers but no
allocator).  Its workspace is a fixed scratch array inside the library, so
this test calls it straight through the C ABI, twice in a row on one stream
with different inputs, and checks each result bit for bit against the
workspace-taking entry point (same kernels, tiles and split order), which a
partial left over from the previous call would break.  It also checks the
size limit at its exact edge and with a split count that fits only after it
is clamped to the K blocks.  It lives in a file of its own that pytest
collects last."""
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
        ref = g.gemm_bf16_nt_splitk(Ad, Bd, splits)
        assert torch.equal(C.view(torch.int16), ref.view(torch.int16)), f"static scratch, {name}"
        check_close16(bits16(C), bits16(ref), K, amax(A), amax(Bh), what=f"static scratch, {name}")
    # and against the oracle, for the second call
    rows = np.arange(0, M, 37)
    check_close16(bits16(C2)[rows], oracle.gemm_bf16_nt(A, B2, rows=rows), K, amax(A), amax(B2),
                  what="static scratch vs oracle")


def test_static_scratch_rejects_problems_over_the_limit(lib):
    # 4 splits of 4096 x 4096 FP32 partials = 256 MiB > the 32 MiB scratch
    P = 0x10000
    assert lib.gemm_bf16_nt_splitk_static(P, 2 * P, 3 * P, 4096, 4096, 4096, 4, None) == 2
    # one 128-row tile over the limit: 2 splits x 2176 x 2048 x 4 bytes
    assert lib.gemm_bf16_nt_splitk_static(P, 2 * P, 3 * P, 2176, 2048, 128, 2, None) == 2


LIMIT = 32 << 20   # GEMM_SPLITK_STATIC_SCRATCH_BYTES


@pytest.mark.parametrize("k_splits", [2, 64], ids=["exact", "clamped"])
def test_static_scratch_at_the_limit(lib, k_splits):
    # 2 effective splits x 2048 x 2048 x 4 bytes = exactly the 32 MiB scratch.
    # K = 128 holds two 64-deep K blocks, so k_splits = 64 is clamped to 2:
    # accepted only because the limit is checked on the splits actually used.
    import nvfp4_block_scaled_tcgen05_gb300 as g
    M, N, K = 2048, 2048, 128
    assert g.gemm_bf16_nt_splitk_workspace_bytes(M, N, K, k_splits) == LIMIT
    A = synth.bf16_normal((M, K), 1.0, 211)
    B = synth.bf16_normal((N, K), 1.0, 212)
    Ad, Bd = to_dev_bf16(A), to_dev_bf16(B)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        C.fill_(float("nan"))
        assert lib.gemm_bf16_nt_splitk_static(Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(),
                                              M, N, K, k_splits, stream) == 0
        ref = g.gemm_bf16_nt_splitk(Ad, Bd, k_splits)
        assert torch.equal(C.view(torch.int16), ref.view(torch.int16))
    assert g.gemm_get_device_status() == 0
