"""GPU parity of the NVFP4 block-scaled GEMM against the oracle: layout
probes with exact expected values (identity operands, one-hot scales),
random small cases spanning several tiles, and the full-size problem on
sampled rows."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import bits16, check_bitexact16, check_close16, sample_rows, to_dev_u8

pytestmark = pytest.mark.gpu
UNIT = 0x38     # e4m3 1.0
ONE = 0x2       # e2m1 1.0
MAXDQ = 6.0 * 4.0  # largest |e2m1 * scale| of the synthetic inputs


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_tcgen05_gb300 as lib
    yield lib
    assert lib.gemm_get_device_status() == 0


@pytest.fixture(params=[2], ids=["cta2"])
def cg(request):
    """The NVFP4 GEMM always runs on CTA pairs (cta_group::2); M = 128
    problems leave the second CTA's rows past M."""
    return request.param


def run(g, a, b, sfa, sfb, L, M, N, K):
    c = g.gemm_nvfp4_bs(to_dev_u8(a), to_dev_u8(b), to_dev_u8(sfa), to_dev_u8(sfb), L, M, N, K)
    return bits16(c).reshape(L * M, N)


def identity_codes(L, rows, K):
    x = np.zeros((L, rows, K // 2), dtype=np.uint8)
    for r in range(min(rows, K)):
        x[:, r, r // 2] |= np.uint8(ONE << (4 * (r % 2)))
    return x


def test_identity_b_gives_dequantised_a(g, cg):
    L, M, N, K = 1, 256, 256, 256
    a, _, sfa, _ = synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, 91))
    b = identity_codes(L, N, K)
    sfb = np.full(L * N * K // 16, UNIT, dtype=np.uint8)
    got = run(g, a, b, sfa, sfb, L, M, N, K)
    check_bitexact16(got, oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K), "identity b",
                     zero_sign=False)


def test_identity_a_gives_dequantised_b_transposed(g, cg):
    L, M, N, K = 1, 256, 384, 256
    _, b, _, sfb = synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, 92))
    a = identity_codes(L, M, K)
    sfa = np.full(L * M * K // 16, UNIT, dtype=np.uint8)
    got = run(g, a, b, sfa, sfb, L, M, N, K)
    check_bitexact16(got, oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K), "identity a")


@pytest.mark.parametrize("side", ["a", "b"])
def test_one_hot_scale(g, cg, side):
    L, M, N, K = 1, 128, 256, 512
    a, b, _, _ = synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, 93))
    sfa = np.full(L * M * K // 16, UNIT, dtype=np.uint8)
    sfb = np.full(L * N * K // 16, UNIT, dtype=np.uint8)
    rest_k = K // 64
    base = run(g, a, b, sfa, sfb, L, M, N, K)
    check_close16(base, oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K), K, 6.0, 6.0, "f16",
                  "unit scales")
    for (r, j) in [(0, 0), (37, 5), (127, 31), (100, 17)] + ([(200, 9)] if side == "b" else []):
        s2a, s2b = sfa.copy(), sfb.copy()
        if side == "a":
            s2a[oracle.sf_offset(r, j, 0, M // 128, rest_k)] = 0x40
        else:
            s2b[oracle.sf_offset(r, j, 0, N // 128, rest_k)] = 0x40
        got = run(g, a, b, s2a, s2b, L, M, N, K)
        ref = oracle.gemm_nvfp4_bs(a, b, s2a, s2b, L, M, N, K)
        check_close16(got, ref, K, 12.0, 6.0, "f16", f"one-hot scale {side} r={r} j={j}")
        changed = np.argwhere(got != base)
        if side == "a":
            assert set(changed[:, 0].tolist()) <= {r}
        else:
            assert set(changed[:, 1].tolist()) <= {r}


@pytest.mark.parametrize("L,M,N,K", [(1, 128, 256, 256), (1, 384, 640, 1024), (2, 256, 384, 512),
                                     (1, 128, 128, 256), (2, 384, 512, 256), (1, 512, 768, 2048)])
def test_random_small(g, cg, L, M, N, K):
    a, b, sfa, sfb = synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, 94 + M + N))
    got = run(g, a, b, sfa, sfb, L, M, N, K)
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K)
    stats = check_close16(got, ref, K, MAXDQ, MAXDQ, "f16", f"nvfp4 {L}x{M}x{N}x{K}")
    assert stats["max_ulp"] <= 1, stats


def test_full_size_sampled(g):
    w = synth.NVFP4
    a, b, sfa, sfb = synth.nvfp4_inputs(w)
    got = run(g, a, b, sfa, sfb, w.L, w.M, w.N, w.K)
    rows = np.array(sorted({0, 1, 31, 32, 127, 128, 2047, 2048, 4064, 4095} |
                           set(np.random.default_rng(9).integers(0, w.M, 22).tolist())))
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, w.L, w.M, w.N, w.K, rows=rows)
    stats = check_close16(got[rows], ref, w.K, MAXDQ, MAXDQ, "f16", "nvfp4 full size")
    assert stats["frac_exact"] > 0.9, stats


# ---------------------------------------------------------------- split-K
def run_splitk(g, a, b, sfa, sfb, M, N, K, k_splits, L=1):
    c = g.gemm_nvfp4_bs_splitk(to_dev_u8(a), to_dev_u8(b), to_dev_u8(sfa), to_dev_u8(sfb),
                               M, N, K, k_splits, L=L)
    return bits16(c).reshape(L * M, N)


@pytest.mark.parametrize("M,N,K,k_splits", [(128, 256, 1024, 3), (256, 512, 2048, 5),
                                            (128, 384, 512, 64), (384, 128, 2304, 4)])
def test_splitk_small(g, M, N, K, k_splits):
    a, b, sfa, sfb = synth.nvfp4_inputs(synth.Nvfp4("t", 1, M, N, K, 97 + M + K))
    got = run_splitk(g, a, b, sfa, sfb, M, N, K, k_splits)
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, 1, M, N, K)
    stats = check_close16(got, ref, K, MAXDQ, MAXDQ, "f16", f"nvfp4 split-K {M}x{N}x{K}/{k_splits}")
    assert stats["max_ulp"] <= 1, stats


@pytest.mark.parametrize("L,M,N,K,k_splits", [
    (2, 128, 512, 1024, 2),     # decode-like: operands swapped, transposed partials
    (3, 256, 384, 2048, 3),     # swapped, two 128-row activation blocks
    (2, 384, 256, 1024, 4),     # M > 256: the unswapped pair kernel
])
def test_splitk_batched(g, L, M, N, K, k_splits):
    a, b, sfa, sfb = synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, 131 + M + L))
    got = run_splitk(g, a, b, sfa, sfb, M, N, K, k_splits, L)
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K)
    stats = check_close16(got, ref, K, MAXDQ, MAXDQ, "f16", f"nvfp4 split-K L={L} {M}x{N}x{K}")
    assert stats["max_ulp"] <= 1, stats


def test_splitk_swapped_exact_and_deterministic(g):
    # integer-valued inputs (codes 0/1/2/3 -> e2m1 0, 0.5, 1, 1.5 with unit
    # scales, exact sums): bit-exact against the oracle, and two runs agree
    L, M, N, K = 1, 128, 768, 4096
    rng = np.random.default_rng(141)
    a = (rng.integers(0, 4, (L, M, K // 2)) | (rng.integers(0, 4, (L, M, K // 2)) << 4)).astype(np.uint8)
    b = (rng.integers(0, 4, (L, N, K // 2)) | (rng.integers(0, 4, (L, N, K // 2)) << 4)).astype(np.uint8)
    sfa = np.full(L * M * K // 16, UNIT, dtype=np.uint8)
    sfb = np.full(L * N * K // 16, UNIT, dtype=np.uint8)
    r1 = run_splitk(g, a, b, sfa, sfb, M, N, K, 5)
    r2 = run_splitk(g, a, b, sfa, sfb, M, N, K, 5)
    assert np.array_equal(r1, r2)
    check_bitexact16(r1, oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K).reshape(M, N),
                     "nvfp4 swapped split-K exact")


def test_splitk_equals_unsplit_within_one_ulp(g):
    M, N, K = 128, 512, 4096
    a, b, sfa, sfb = synth.nvfp4_inputs(synth.Nvfp4("t", 1, M, N, K, 98))
    whole = run(g, a, b, sfa, sfb, 1, M, N, K)
    split = run_splitk(g, a, b, sfa, sfb, M, N, K, 4)
    d = np.abs(whole.astype(np.int32) - split.astype(np.int32))
    assert d.max() <= 1, d.max()


@pytest.mark.parametrize("name", sorted(synth.NVFP4_DECODE))
def test_splitk_decode_shapes_sampled(g, name):
    w, k_splits = synth.NVFP4_DECODE[name]
    a, b, sfa, sfb = synth.nvfp4_inputs(w)
    got = run_splitk(g, a, b, sfa, sfb, w.M, w.N, w.K, k_splits)
    rows = np.array([0, 1, 31, 32, 63, 64, 100, 127])
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, w.L, w.M, w.N, w.K, rows=rows)
    stats = check_close16(got[rows], ref, w.K, MAXDQ, MAXDQ, "f16", name)
    assert stats["frac_exact"] > 0.9, stats


def test_splitk_workspace_is_not_read(g):
    # stale workspace contents must not leak into the result
    M, N, K = 128, 256, 1024
    a, b, sfa, sfb = synth.nvfp4_inputs(synth.Nvfp4("t", 1, M, N, K, 99))
    need = g.gemm_nvfp4_bs_splitk_workspace_bytes(M, N, K, 4)
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device="cuda")
    c = g.gemm_nvfp4_bs_splitk(to_dev_u8(a), to_dev_u8(b), to_dev_u8(sfa), to_dev_u8(sfb),
                               M, N, K, 4, workspace=ws)
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, 1, M, N, K)
    check_close16(bits16(c).reshape(M, N), ref, K, MAXDQ, MAXDQ, "f16", "stale workspace")


@pytest.mark.parametrize("fill", [0x00, 0x7F, 0xFF])
def test_splitk_any_workspace_contents_same_result(g, fill):
    # batched decode-like split-K: whatever the workspace holds on entry, the
    # result equals the one from a fresh workspace bit for bit
    L, M, N, K = 2, 128, 512, 2048
    a, b, sfa, sfb = synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, 171))
    args = [to_dev_u8(x) for x in (a, b, sfa, sfb)]
    need = L * g.gemm_nvfp4_bs_splitk_workspace_bytes(M, N, K, 4)
    ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
    got = bits16(g.gemm_nvfp4_bs_splitk(*args, M, N, K, 4, workspace=ws, L=L)).reshape(L * M, N)
    fresh = bits16(g.gemm_nvfp4_bs_splitk(*args, M, N, K, 4, L=L)).reshape(L * M, N)
    assert np.array_equal(got, fresh)
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K)
    check_close16(got, ref, K, MAXDQ, MAXDQ, "f16", f"workspace fill {fill:#x}")


def test_splitk_graph_replay(g):
    # the GEMM and its reduce captured in one graph and replayed with new
    # activations each time
    M, N, K, S = 128, 768, 4096, 4
    a, b, sfa, sfb = synth.nvfp4_inputs(synth.Nvfp4("t", 1, M, N, K, 181))
    ad, bd, sad, sbd = [to_dev_u8(x) for x in (a, b, sfa, sfb)]
    need = g.gemm_nvfp4_bs_splitk_workspace_bytes(M, N, K, S)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    c = torch.empty((1, M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g.gemm_nvfp4_bs_splitk(ad, bd, sad, sbd, M, N, K, S, workspace=ws, c=c, stream=s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.gemm_nvfp4_bs_splitk(ad, bd, sad, sbd, M, N, K, S, workspace=ws, c=c, stream=s)
    for seed in (182, 183, 184):
        a2 = synth.nvfp4_inputs(synth.Nvfp4("t", 1, M, N, K, seed))[0]
        ad.copy_(to_dev_u8(a2))
        c.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.gemm_nvfp4_bs(a2, b, sfa, sfb, 1, M, N, K)
        check_close16(bits16(c).reshape(M, N), ref, K, MAXDQ, MAXDQ, "f16", f"replay {seed}")


def test_splitk_back_to_back_shares_workspace(g):
    # launches of different shapes and split counts queued on one stream
    # without synchronisation, sharing one workspace (each GEMM's partials
    # are read by its own reduce before the next GEMM writes them)
    cases = [(1, 128, 512, 2048, 4), (2, 256, 256, 1024, 2), (1, 128, 768, 4096, 3)]
    need = max(L * g.gemm_nvfp4_bs_splitk_workspace_bytes(M, N, K, S) for L, M, N, K, S in cases)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    inputs = [synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, 191 + i))
              for i, (L, M, N, K, S) in enumerate(cases)]
    devs = [[to_dev_u8(x) for x in inp] for inp in inputs]
    outs = []
    torch.cuda.synchronize()
    for rep in range(3):
        for (L, M, N, K, S), d in zip(cases, devs):
            outs.append(g.gemm_nvfp4_bs_splitk(*d, M, N, K, S, workspace=ws, L=L))
    torch.cuda.synchronize()
    for i, (L, M, N, K, S) in enumerate(cases):
        a, b, sfa, sfb = inputs[i]
        ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K)
        first = bits16(outs[i]).reshape(L * M, N)
        check_close16(first, ref, K, MAXDQ, MAXDQ, "f16", f"back to back {L}x{M}x{N}x{K}/{S}")
        for rep in (1, 2):
            assert np.array_equal(bits16(outs[rep * len(cases) + i]).reshape(L * M, N), first)
