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


def _bits_equal_nan_aware(got, ref, what):
    # NaN payloads may differ between the oracle and the device; every other
    # value, signed zeros and infinities included, must match bit for bit
    gb, rb = got.view(np.uint32), ref.view(np.uint32)
    both_nan = np.isnan(got) & np.isnan(ref)
    bad = (gb != rb) & ~both_nan
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} differ; first {idx.tolist()}")


@pytest.mark.parametrize("special", ["tiny", "subnormal", "huge", "inf_nan"])
def test_router_slices_outside_the_fused_range(g, special):
    # N(0,1) operands with a few values outside [2^-63, 2^63) planted in some
    # 16-deep K slices of some 64-row / 64-column blocks: those slices run
    # separate multiplies and adds, the rest fused multiply-adds; every
    # output must still equal the strict loop's bit for bit
    M, N, K = 200, 136, 160
    A = synth.bf16_normal((M, K), 1.0, 301)
    B = synth.bf16_normal((N, K), 1.0, 302)
    rng = np.random.default_rng(303)
    vals = {"tiny": [0x1A00, 0x9A80, 0x1F00],        # 2^-75, -2^-74, 2^-65
            "subnormal": [0x0001, 0x8040, 0x007F],   # bf16 subnormals
            "huge": [0x6000, 0xE100, 0x7F7F],        # 2^65, -2^67, max finite
            "inf_nan": [0x7F80, 0xFF80, 0x7FC0]}[special]
    for _ in range(6):
        r, k = int(rng.integers(0, M)), int(rng.integers(0, K))
        A[r, k] = vals[int(rng.integers(0, len(vals)))]
        n, k2 = int(rng.integers(0, N)), int(rng.integers(0, K))
        B[n, k2] = vals[int(rng.integers(0, len(vals)))]
    _bits_equal_nan_aware(router(g, A, B), oracle.gemm_router(A, B), f"router {special}")


def test_router_tiny_products_in_every_slice_position(g):
    # the golden subnormal-tie sequence placed at K offsets 0..47 (three
    # slices), surrounded by ordinary values: exact wherever it falls
    M, N, K = 64, 64, 64
    base_a = synth.bf16_normal((M, K), 1.0, 311)
    base_b = synth.bf16_normal((N, K), 1.0, 312)
    seq_a, seq_b = [0x2000, 0x1A00, 0x1AC0], [0x2000, 0x1A80, 0x1A00]
    for off in range(0, 46, 5):
        A, B = base_a.copy(), base_b.copy()
        A[3, :] = 0
        B[5, :] = 0
        A[3, off:off + 3] = seq_a
        B[5, off:off + 3] = seq_b
        got = router(g, A, B)
        assert_bits_equal(got, oracle.gemm_router(A, B), f"tie sequence at k={off}")
        assert got.view(np.uint32)[3, 5] == 0x00800003
