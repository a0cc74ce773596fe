"""GPU parity of the split-K BF16 GEMM (FP32 partials in a caller workspace,
fixed-order reduce) against the oracle."""
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
    """Force the single-CTA or the CTA-pair split-K kernel."""
    g.gemm_testing_set_overrides(cta_group=request.param)
    yield request.param
    g.gemm_testing_set_overrides()


def amax(x):
    return float(np.abs(bf16_val(x)).max())


@pytest.mark.parametrize("M,N,K,splits", [(300, 520, 200, 3), (128, 256, 2048, 4),
                                          (640, 512, 1032, 5), (129, 264, 72, 2), (256, 512, 640, 1)])
def test_splitk_ragged(g, cg, M, N, K, splits):
    A = synth.bf16_normal((M, K), 1.0, 101 + M)
    B = synth.bf16_normal((N, K), 1.0, 102 + N)
    C = g.gemm_bf16_nt_splitk(to_dev_bf16(A), to_dev_bf16(B), splits)
    check_close16(bits16(C), oracle.gemm_bf16_nt(A, B), K, amax(A), amax(B),
                  what=f"splitk {M}x{N}x{K}/{splits}")


def test_splitk_exact_integers_and_determinism(g, cg):
    M, N, K = 384, 512, 1024
    A = synth.bf16_small_ints((M, K), -3, 3, 111)
    B = synth.bf16_small_ints((N, K), -3, 3, 112)
    Ad, Bd = to_dev_bf16(A), to_dev_bf16(B)
    C1 = bits16(g.gemm_bf16_nt_splitk(Ad, Bd, 4))
    C2 = bits16(g.gemm_bf16_nt_splitk(Ad, Bd, 4))
    assert np.array_equal(C1, C2)
    check_bitexact16(C1, oracle.gemm_bf16_nt(A, B), "splitk exact integers")


def test_splitk_gqa_full_size_sampled(g):
    w = synth.BF16_WORKLOADS["gqa"]
    A, B = synth.gemm_inputs(w)
    C = bits16(g.gemm_bf16_nt_splitk(to_dev_bf16(A), to_dev_bf16(B), 4))
    rows = sample_rows(w.M, n_random=64, seed=7)
    check_close16(C[rows], oracle.gemm_bf16_nt(A, B, rows=rows), w.K, amax(A), amax(B),
                  what="gqa splitk")


def test_splitk_workspace_too_small(g):
    A = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.GemmError) as e:
        g.gemm_bf16_nt_splitk(A, B, 2, workspace=ws)
    assert e.value.status == 2
