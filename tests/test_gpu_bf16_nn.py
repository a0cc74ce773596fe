"""GPU parity of the NN-layout BF16 GEMM (B stored [K][N]) against the CPU
oracle (the plain definition C = A.B evaluated by the NT oracle on B^T), and
its bit-equality with the NT kernel on the transposed operand."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import bf16_val, bits16, check_bitexact16, check_close16, sample_rows, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_tcgen05_gb300 as lib
    yield lib
    assert lib.gemm_get_device_status() == 0


@pytest.fixture(params=[1, 2], ids=["cta1", "cta2"])
def cg(request, g):
    """Force the single-CTA or the CTA-pair kernel."""
    g.gemm_testing_set_overrides(cta_group=request.param)
    yield request.param
    g.gemm_testing_set_overrides()


def amax(x):
    return float(np.abs(bf16_val(x)).max())


def nn(g, A, Bkn):
    return bits16(g.gemm_bf16_nn(to_dev_bf16(A), to_dev_bf16(Bkn)))


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 256),     # one tile
    (300, 520, 200),     # ragged M, N and K tail
    (1, 8, 8),           # degenerate
    (129, 264, 72),      # one row / 8 columns past a tile, K tail of 8
    (17, 1000, 1032),    # many K blocks with a tail
    (640, 768, 64),      # exact multiples
])
def test_gemm_bf16_nn_ragged(g, cg, M, N, K):
    A = synth.bf16_normal((M, K), 1.0, 211 + M)
    Bkn = synth.bf16_normal((K, N), 1.0, 212 + N)
    got = nn(g, A, Bkn)
    ref = oracle.gemm_bf16_nt(A, np.ascontiguousarray(Bkn.T))
    check_close16(got, ref, K, amax(A), amax(Bkn), what=f"nn {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(256, 512, 1024), (300, 520, 200)])
def test_gemm_bf16_nn_equals_nt_on_transposed_b(g, cg, M, N, K):
    A = synth.bf16_normal((M, K), 1.0, 221 + M)
    Bkn = synth.bf16_normal((K, N), 1.0, 222 + N)
    got = nn(g, A, Bkn)
    nt = bits16(g.gemm_bf16_nt(to_dev_bf16(A), to_dev_bf16(np.ascontiguousarray(Bkn.T))))
    check_bitexact16(got, nt, "nn vs nt(B^T)")


def test_gemm_bf16_nn_identity_and_selection(g, cg):
    M, K = 256, 384
    A = synth.bf16_normal((M, K), 1.0, 231)
    eye = np.zeros((K, K), dtype=np.uint16)
    eye[np.arange(K), np.arange(K)] = 0x3F80
    check_bitexact16(nn(g, A, eye), A, "identity B")
    # B picks columns: C[:, n] = A[:, perm[n]]
    perm = np.random.default_rng(5).permutation(K)[:136]
    P = np.zeros((K, 136), dtype=np.uint16)
    P[perm, np.arange(136)] = 0x3F80
    check_bitexact16(nn(g, A, P), A[:, perm], "column selection")


def test_gemm_bf16_nn_full_size_sampled(g):
    w = synth.BF16_WORKLOADS["gateup"]
    A, B = synth.gemm_inputs(w)          # B [N][K]; the NN operand is its transpose
    Bkn = np.ascontiguousarray(B.T)
    got = nn(g, A, Bkn)
    rows = sample_rows(w.M, n_random=32, seed=7)
    ref = oracle.gemm_bf16_nt(A, B, rows=rows)
    stats = check_close16(got[rows], ref, w.K, amax(A), amax(B), what="nn gate/up")
    assert stats["frac_exact"] > 0.9, stats
