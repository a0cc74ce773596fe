"""GPU parity of the ordered FP32 router GEMM: bit-exact against the oracle's
strict sequential, FMA-free loop."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import to_dev_bf16

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_tcgen05_gb300 as lib
    yield lib
    assert lib.gemm_get_device_status() == 0


def router(g, A, B):
    C = g.gemm_bf16_nt_ordered(to_dev_bf16(A), to_dev_bf16(B))
    return C.cpu().numpy()


def assert_bits_equal(got, ref, what):
    gb, rb = got.view(np.uint32), ref.view(np.uint32)
    if not np.array_equal(gb, rb):
        idx = np.argwhere(gb != rb)[:5]
        raise AssertionError(f"{what}: {int((gb != rb).sum())} differ; first {idx.tolist()}")


def test_router_full_config_bitexact(g):
    w = synth.ROUTER
    A, B = synth.gemm_inputs(w)
    assert_bits_equal(router(g, A, B), oracle.gemm_router(A, B), "router 4510x256x2048")


@pytest.mark.parametrize("M,N,K", [(1, 1, 8), (65, 70, 40), (2255, 256, 2048), (100, 3, 1000)])
def test_router_ragged_bitexact(g, M, N, K):
    A = synth.bf16_normal((M, K), 1.0, 81 + M)
    B = synth.bf16_normal((N, K), 1.0, 82 + N)
    assert_bits_equal(router(g, A, B), oracle.gemm_router(A, B), f"router {M}x{N}x{K}")


def test_router_fma_and_subnormal_golden(g):
    with open(os.path.join(GOLDEN, "router_fma_case.txt")) as f:
        vals = {ln.split()[0]: [int(v, 16) for v in ln.split()[1:]]
                for ln in f if ln.strip() and not ln.startswith("#")}
    # pad K to a multiple of 8 with zero products at the end (acc + 0 = acc)
    A = np.zeros((1, 8), dtype=np.uint16)
    B = np.zeros((1, 8), dtype=np.uint16)
    A[0, :3] = vals["a_bf16"]
    B[0, :3] = vals["b_bf16"]
    got = router(g, A, B).view(np.uint32)
    assert got[0, 0] == vals["c_f32"][0], hex(got[0, 0])


def test_router_signed_zero_and_cancellation(g):
    K = 16
    A = np.zeros((3, K), dtype=np.uint16)
    A[1] = 0x8000                          # -0 row
    A[2, :3] = [0x4B80, 0x3F80, 0xCB80]    # 2^24, 1, -2^24
    B = np.zeros((2, K), dtype=np.uint16)
    B[0, :3] = 0x3F80
    B[1] = 0xBF80                          # -1 everywhere
    got = router(g, A, B)
    assert_bits_equal(got, oracle.gemm_router(A, B), "signed zero / cancellation")
    assert got.view(np.uint32)[1, 1] == 0  # +0, never -0
