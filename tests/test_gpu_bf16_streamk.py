"""GPU parity of the stream-K BF16 NT GEMM against the CPU oracle, through the
C ABI: whole tiles equal the data-parallel GEMM bit for bit; tiles whose K
iterations were divided over several CTA pairs are the ordered FP32 sum of
their partial tiles, within the GEMM tolerance of the oracle (bit-exact where
every partial sum is an exact integer)."""
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


@pytest.fixture(params=["all", "5"], ids=["share_all", "share_5"])
def share(request, g):
    """Force the stream-K division of the tail over every CTA pair, or over
    five pairs (several segments per pair); by default the library divides
    the tail only when it leaves most pairs idle."""
    g.gemm_testing_set_overrides(streamk_clusters=4096 if request.param == "all" else 5)
    yield request.param
    g.gemm_testing_set_overrides()


@pytest.fixture(scope="module")
def ws(g):
    n = g.gemm_bf16_nt_streamk_workspace_bytes()
    assert n > 0
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def amax(x):
    return float(np.abs(bf16_val(x)).max())


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 256),     # one tile, two 128-deep K iterations on two pairs
    (300, 520, 200),     # ragged M, N and K tail; every tile split
    (1, 8, 8),           # one iteration: one pair stores the whole tile
    (129, 264, 72),      # one row / 8 columns past a tile
    (17, 1000, 1032),    # 4 tiles x 9 iterations over the pairs
    (2048, 4096, 1032),  # 128 tiles: a data-parallel round, then a split tail
])
def test_streamk_ragged(g, ws, share, M, N, K):
    A = synth.bf16_normal((M, K), 1.0, 11 + M)
    B = synth.bf16_normal((N, K), 1.0, 12 + N)
    C = g.gemm_bf16_nt_streamk(to_dev_bf16(A), to_dev_bf16(B), ws)
    rows = np.arange(M) if M <= 512 else sample_rows(M, n_random=64, seed=M)
    ref = oracle.gemm_bf16_nt(A, B, rows=rows)
    check_close16(bits16(C)[rows], ref, K, amax(A), amax(B), what=f"stream-K {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(384, 520, 512), (2048, 4096, 1032), (4096, 2048, 2048)])
def test_streamk_exact_integers_bitexact(g, ws, share, M, N, K):
    # every partial and every sum of partials is an exact FP32 integer, so the
    # split tiles must round to exactly the oracle's values
    A = synth.bf16_small_ints((M, K), -3, 3, 21 + K)
    B = synth.bf16_small_ints((N, K), -3, 3, 22 + K)
    C = g.gemm_bf16_nt_streamk(to_dev_bf16(A), to_dev_bf16(B), ws)
    check_bitexact16(bits16(C), oracle.gemm_bf16_nt(A, B), f"stream-K exact {M}x{N}x{K}")


def test_streamk_whole_tiles_equal_data_parallel(g, ws):
    # qkv shape: 160 tiles, a tail of 8 on 76 pairs, which the default
    # schedule divides; all but the tail round are whole-tile work
    g.gemm_testing_set_overrides()
    w = synth.BF16_WORKLOADS["qkv"]
    A, B = synth.gemm_inputs(w)
    Ad, Bd = to_dev_bf16(A), to_dev_bf16(B)
    sk = bits16(g.gemm_bf16_nt_streamk(Ad, Bd, ws)).reshape(w.M // 256, 256, w.N // 256, 256)
    dp = bits16(g.gemm_bf16_nt(Ad, Bd)).reshape(w.M // 256, 256, w.N // 256, 256)
    same = (sk == dp).all(axis=(1, 3))
    # 160 tiles on at most 76 pairs: the two data-parallel rounds (152 tiles
    # when all 76 pairs are co-resident) are bit-identical to the plain GEMM
    assert same.sum() >= 0.9 * same.size, int(same.sum())


def test_streamk_stale_workspace_and_determinism(g, ws, share):
    M, N, K = 1000, 1032, 776
    A = synth.bf16_normal((M, K), 1.0, 81)
    B = synth.bf16_normal((N, K), 1.0, 82)
    Ad, Bd = to_dev_bf16(A), to_dev_bf16(B)
    ws.view(torch.float32).fill_(float("nan"))
    C1 = bits16(g.gemm_bf16_nt_streamk(Ad, Bd, ws))
    ws.view(torch.float32).fill_(-1.0e30)
    C2 = bits16(g.gemm_bf16_nt_streamk(Ad, Bd, ws))
    assert np.array_equal(C1, C2)
    check_close16(C1, oracle.gemm_bf16_nt(A, B), K, amax(A), amax(B), what="stale workspace")


def test_streamk_no_write_outside_c(g, ws, share):
    M, N, K = 200, 264, 520
    A = synth.bf16_normal((M, K), 1.0, 91)
    B = synth.bf16_normal((N, K), 1.0, 92)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    C = buf[guard:guard + M * N].view(M, N)
    g.gemm_bf16_nt_streamk(to_dev_bf16(A), to_dev_bf16(B), ws, C)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + M * N:] == 7.0)
    check_close16(bits16(C), oracle.gemm_bf16_nt(A, B), K, amax(A), amax(B), what="guarded")


@pytest.mark.parametrize("name", ["qkv", "gqa"])
def test_streamk_full_size_sampled(g, ws, name):
    w = synth.BF16_WORKLOADS[name]
    A, B = synth.gemm_inputs(w)
    C = bits16(g.gemm_bf16_nt_streamk(to_dev_bf16(A), to_dev_bf16(B), ws))
    rows = sample_rows(w.M, n_random=64, seed=7)
    ref = oracle.gemm_bf16_nt(A, B, rows=rows)
    stats = check_close16(C[rows], ref, w.K, amax(A), amax(B), what=f"stream-K {name}")
    assert stats["frac_exact"] > 0.9, stats


def test_streamk_rejects_a_small_workspace(g, ws):
    A = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GemmError):
        g.gemm_bf16_nt_streamk(A, B, ws[:1024])


def _random_shapes(seed, count):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(1, 1600)), int(rng.integers(1, 260)) * 8, int(rng.integers(1, 400)) * 8)
            for _ in range(count)]


@pytest.mark.parametrize("M,N,K", _random_shapes(2024, 6))
def test_streamk_random_shapes_exact_integers(g, ws, share, M, N, K):
    # seeded ragged shapes, every sum an exact integer: bit-exact for any
    # division of the tail
    A = synth.bf16_small_ints((M, K), -2, 2, M + 3 * K)
    B = synth.bf16_small_ints((N, K), -2, 2, N + 5 * K)
    C = g.gemm_bf16_nt_streamk(to_dev_bf16(A), to_dev_bf16(B), ws)
    check_bitexact16(bits16(C), oracle.gemm_bf16_nt(A, B), f"stream-K random {M}x{N}x{K}")
