"""GPU parity of the BF16 NT GEMM and the fused scaled-acc epilogue against
the CPU oracle, through the C ABI (torch only provides device memory)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import (bf16_val, bits16, check_bitexact16, check_close16, check_scaled_acc,
                    sample_rows, to_dev_bf16)

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
    """Force the single-CTA kernel or the CTA-pair (cta_group::2) kernel."""
    g.gemm_testing_set_overrides(cta_group=request.param)
    yield request.param
    g.gemm_testing_set_overrides()


def amax(x):
    return float(np.abs(bf16_val(x)).max())


def run_gemm(g, A, B):
    C = g.gemm_bf16_nt(to_dev_bf16(A), to_dev_bf16(B))
    return bits16(C)


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 256),     # one tile
    (300, 520, 200),     # ragged M, N and K tail
    (1, 8, 8),           # degenerate
    (129, 264, 72),      # one row / 8 columns past a tile, K tail of 8
    (17, 1000, 1032),    # many K blocks with a tail
    (640, 768, 64),      # exact multiples
])
def test_gemm_bf16_ragged(g, cg, M, N, K):
    A = synth.bf16_normal((M, K), 1.0, 11 + M)
    B = synth.bf16_normal((N, K), 1.0, 12 + N)
    got = run_gemm(g, A, B)
    ref = oracle.gemm_bf16_nt(A, B)
    check_close16(got, ref, K, amax(A), amax(B), what=f"gemm {M}x{N}x{K}")


def test_gemm_bf16_exact_integers_bitexact(g, cg):
    M, N, K = 384, 520, 512
    A = synth.bf16_small_ints((M, K), -3, 3, 21)
    B = synth.bf16_small_ints((N, K), -3, 3, 22)
    check_bitexact16(run_gemm(g, A, B), oracle.gemm_bf16_nt(A, B), "exact integers")


def test_gemm_bf16_identity_and_permutation(g, cg):
    M, K = 300, 256
    A = synth.bf16_normal((M, K), 1.0, 23)
    eye = np.zeros((K, K), dtype=np.uint16)
    eye[np.arange(K), np.arange(K)] = 0x3F80
    check_bitexact16(run_gemm(g, A, eye), A, "identity", zero_sign=False)
    perm = np.random.default_rng(1).permutation(K)
    P = np.zeros((K, K), dtype=np.uint16)
    P[np.arange(K), perm] = 0x3F80
    check_bitexact16(run_gemm(g, A, P), A[:, perm], "permutation")


def test_gemm_bf16_many_tiles_per_cta(g, cg):
    # 32 x 16 = 512 tiles: every CTA walks several tiles and both TMEM buffers
    M, N, K = 4096, 4096, 128
    A = synth.bf16_normal((M, K), 1.0, 31)
    B = synth.bf16_normal((N, K), 1.0, 32)
    got = run_gemm(g, A, B)
    rows = sample_rows(M, n_random=64, seed=3)
    ref = oracle.gemm_bf16_nt(A, B, rows=rows)
    check_close16(got[rows], ref, K, amax(A), amax(B), what="many tiles")


def test_gemm_bf16_no_write_outside_c(g, cg):
    M, N, K = 200, 264, 64
    A = synth.bf16_normal((M, K), 1.0, 41)
    B = synth.bf16_normal((N, K), 1.0, 42)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    C = buf[guard:guard + M * N].view(M, N)
    g.gemm_bf16_nt(to_dev_bf16(A), to_dev_bf16(B), C)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + M * N:] == 7.0)
    check_close16(bits16(C), oracle.gemm_bf16_nt(A, B), K, amax(A), amax(B), what="guarded")


@pytest.mark.parametrize("name", ["gateup", "down", "qkv", "gqa"])
def test_gemm_bf16_full_size_sampled(g, name):
    w = synth.BF16_WORKLOADS[name]
    A, B = synth.gemm_inputs(w)
    got = run_gemm(g, A, B)
    rows = sample_rows(w.M, n_random=64, seed=5)
    ref = oracle.gemm_bf16_nt(A, B, rows=rows)
    stats = check_close16(got[rows], ref, w.K, amax(A), amax(B), what=name)
    assert stats["frac_exact"] > 0.9, stats


# ---------------------------------------------------------------- scaled-acc

def test_scaled_acc_tiny_config(g):
    w = synth.BF16_WORKLOADS["tiny"]
    A, B = synth.gemm_inputs(w)
    out0 = synth.scaled_acc_out(w.M, w.N, w.seed)
    O = to_dev_bf16(out0)
    g.gemm_bf16_nt_scaled_acc(to_dev_bf16(A), to_dev_bf16(B), O, synth.TINY_SCALE)
    ref = oracle.gemm_bf16_nt_scaled_acc(A, B, out0, synth.TINY_SCALE)
    d = oracle.gemm_bf16_nt(A, B)
    check_scaled_acc(bits16(O), ref, d, synth.TINY_SCALE, w.K, amax(A), amax(B), "tiny scaled-acc")


@pytest.mark.parametrize("M,N,K,scale", [(128, 256, 256, 0.5), (300, 520, 200, 2.0),
                                         (257, 1032, 16, -0.375), (64, 64, 24, 1.0)])
def test_scaled_acc_fused_equals_unfused_bitexact(g, cg, M, N, K, scale):
    A = synth.bf16_normal((M, K), 1.0, 51 + K)
    B = synth.bf16_normal((N, K), 0.5, 52 + K)
    out0 = synth.bf16_normal((M, N), 1.0, 53 + K)
    Ad, Bd = to_dev_bf16(A), to_dev_bf16(B)
    fused = to_dev_bf16(out0)
    g.gemm_bf16_nt_scaled_acc(Ad, Bd, fused, scale)
    scratch = g.gemm_bf16_nt(Ad, Bd)
    unfused = to_dev_bf16(out0)
    g.bf16_scaled_add(unfused, scratch, scale)
    check_bitexact16(bits16(fused), bits16(unfused), "fused vs unfused", zero_sign=True)
    ref = oracle.gemm_bf16_nt_scaled_acc(A, B, out0, scale)
    check_close16(bits16(scratch), oracle.gemm_bf16_nt(A, B), K, amax(A), amax(B), what="delta")
    check_scaled_acc(bits16(fused), ref, oracle.gemm_bf16_nt(A, B), scale, K, amax(A), amax(B),
                     "scaled-acc")


def test_scaled_acc_lora_full_config(g):
    w = synth.LORA
    X, W = synth.gemm_inputs(w)
    out0 = synth.scaled_acc_out(w.M, w.N, w.seed)
    Xd, Wd = to_dev_bf16(X), to_dev_bf16(W)
    O = to_dev_bf16(out0)
    g.gemm_bf16_nt_scaled_acc(Xd, Wd, O, synth.LORA_SCALE)
    got = bits16(O)
    ref = oracle.gemm_bf16_nt_scaled_acc(X, W, out0, synth.LORA_SCALE)
    d_ref = oracle.gemm_bf16_nt(X, W)
    stats = check_scaled_acc(got, ref, d_ref, synth.LORA_SCALE, w.K, amax(X), amax(W), "lora")
    assert stats["frac_exact"] > 0.99, stats
    D = g.gemm_bf16_nt(Xd, Wd)
    check_close16(bits16(D), d_ref, w.K, amax(X), amax(W), what="lora delta")
    unfused = to_dev_bf16(out0)
    g.bf16_scaled_add(unfused, D, synth.LORA_SCALE)
    check_bitexact16(got, bits16(unfused), "lora fused vs unfused", zero_sign=True)


def test_scaled_add_matches_oracle_bitexact(g):
    n = 1_000_003  # odd length: vector body plus scalar tail
    out0 = synth.bf16_normal((n,), 1.0, 61)
    d = synth.bf16_normal((n,), 1.0, 62)
    O = to_dev_bf16(out0)
    g.bf16_scaled_add(O, to_dev_bf16(d), -1.75)
    check_bitexact16(bits16(O), oracle.bf16_scaled_add(out0, d, -1.75), "scaled_add",
                     zero_sign=True)


def test_back_to_back_calls_on_a_side_stream(g):
    M, N, K = 512, 1024, 256
    A = synth.bf16_normal((M, K), 1.0, 71)
    B = synth.bf16_normal((N, K), 1.0, 72)
    Ad, Bd = to_dev_bf16(A), to_dev_bf16(B)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(3):
            outs.append(g.gemm_bf16_nt(Ad, Bd, stream=s))
    s.synchronize()
    ref = oracle.gemm_bf16_nt(A, B)
    for C in outs:
        check_close16(bits16(C), ref, K, amax(A), amax(B), what="side stream")
    assert np.array_equal(bits16(outs[0]), bits16(outs[2]))  # deterministic
