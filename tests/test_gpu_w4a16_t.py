"""GPU parity of the W4A16 GEMM with the weights in the transposed NVFP4
layout ("gemm_dense.rs", w4a16_gemm_n128_ldb / w4a16_gemm_n128_m128_bf16:
transposed-B rows ldb bytes apart, ldb = align_up(N, 128) for odd N) against
the CPU oracle, through the C ABI.  The padding columns hold junk, which must
not reach C."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import bf16_val, bits16, check_bitexact16, check_close16, sample_rows, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_tcgen05_gb300 as lib
    yield lib
    assert lib.gemm_get_device_status() == 0


def align_up(x, a):
    return -(-x // a) * a


def transposed(b, sfb, ldb, seed):
    """The row-layout code and scale bytes transposed into [K/2][ldb] and
    [K/16][ldb], padding columns filled with random junk."""
    rng = np.random.default_rng(seed)
    N = b.shape[0]
    b_t = rng.integers(0, 256, (b.shape[1], ldb), dtype=np.uint8)
    sfb_t = rng.integers(0, 256, (sfb.shape[1], ldb), dtype=np.uint8)
    b_t[:, :N] = b.T
    sfb_t[:, :N] = sfb.T
    return b_t, sfb_t


def run(g, A, b_t, sfb_t, scale2, N):
    return bits16(g.gemm_w4a16_t(to_dev_bf16(A), to_dev_u8(b_t), to_dev_u8(sfb_t), scale2, N))


def wmax(b, sfb, scale2):
    tab = np.abs(np.array(E2M1))
    hi = np.maximum(tab[b & 0xF], tab[b >> 4]).reshape(b.shape[0], -1, 8).max(axis=2)
    sc = torch.from_numpy(sfb.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return float((hi * sc).max() * abs(scale2))


def amax(x):
    return float(np.abs(bf16_val(x)).max())


def w4_inputs(M, N, K, seed, scale2=0.37):
    A = synth.bf16_normal((M, K), 1.0, seed)
    b = synth.uniform_bytes(N * K // 2, seed + 1).reshape(N, K // 2)
    sfb = synth.e4m3_range_bytes(N * K // 16, seed + 2).reshape(N, K // 16)
    return A, b, sfb, float(np.float32(scale2))


@pytest.mark.parametrize("M,N,K,ldb", [
    (128, 256, 256, 256),      # one tile, packed rows (ldb = N)
    (300, 521, 768, 640),      # odd N padded to align_up(N, 128); ragged M
    (1, 1, 128, 16),           # degenerate: one column, one K block
    (129, 263, 512, 384),      # one row past a tile; odd N
    (17, 1000, 2304, 1024),    # many stages, N not a multiple of 256
    (640, 768, 128, 784),      # exact multiples, a stride that is not a multiple of 128
])
def test_w4a16_t_ragged(g, M, N, K, ldb):
    A, b, sfb, scale2 = w4_inputs(M, N, K, 600 + M + N)
    b_t, sfb_t = transposed(b, sfb, ldb, 601 + N)
    got = run(g, A, b_t, sfb_t, scale2, N)
    ref = oracle.gemm_w4a16_t(A, b_t, sfb_t, scale2, N)
    check_close16(got, ref, K, amax(A), wmax(b, sfb, scale2), what=f"w4a16_t {M}x{N}x{K} ldb={ldb}")


@pytest.mark.parametrize("M,N,K,ldb", [(384, 519, 512, 640), (256, 256, 2048, 256), (77, 131, 256, 144)])
def test_w4a16_t_exact_integers_bitexact(g, M, N, K, ldb):
    # block scales 2.0 make every weight a small integer; small-integer
    # activations keep every FP32 sum exact: bit-exact
    A = synth.bf16_small_ints((M, K), -3, 3, 71 + K)
    b = synth.uniform_bytes(N * K // 2, 72 + K).reshape(N, K // 2)
    sfb = np.full((N, K // 16), 0x40, dtype=np.uint8)
    b_t, sfb_t = transposed(b, sfb, ldb, 73)
    got = run(g, A, b_t, sfb_t, 0.25, N)
    check_bitexact16(got, oracle.gemm_w4a16_t(A, b_t, sfb_t, 0.25, N),
                     f"w4a16_t exact {M}x{N}x{K}")


def test_w4a16_t_identity_reads_back_every_weight(g):
    # A = I: C[m, n] = w[n, m] (one product per output): every dequantised
    # weight, nibble and scale placement comes back bit for bit
    K, N, ldb = 256, 263, 384
    A = np.zeros((K, K), dtype=np.uint16)
    A[np.arange(K), np.arange(K)] = 0x3F80
    b = synth.uniform_bytes(N * K // 2, 81).reshape(N, K // 2)
    sfb = synth.e4m3_range_bytes(N * K // 16, 82, 0x01, 0x7E).reshape(N, K // 16)
    b_t, sfb_t = transposed(b, sfb, ldb, 83)
    for scale2 in (1.0, -3.7):
        check_bitexact16(run(g, A, b_t, sfb_t, scale2, N),
                         oracle.gemm_w4a16_t(A, b_t, sfb_t, scale2, N), f"identity {scale2}")


@pytest.mark.parametrize("M,N,K", [(300, 520, 768), (1016, 1024, 2048), (129, 264, 512)])
def test_w4a16_t_equals_row_layout_kernel(g, M, N, K):
    # same tiles and MMA sequence as gemm_w4a16 (B staged MN-major instead of
    # K-major): bit-identical on the same weights
    A, b, sfb, scale2 = w4_inputs(M, N, K, 700 + M)
    b_t, sfb_t = transposed(b, sfb, align_up(N, 128), 701)
    rows = bits16(g.gemm_w4a16(to_dev_bf16(A), to_dev_u8(b), to_dev_u8(sfb), scale2))
    check_bitexact16(run(g, A, b_t, sfb_t, scale2, N), rows, f"transposed vs rows {M}x{N}x{K}")


def test_w4a16_t_no_write_outside_c(g):
    M, N, K, ldb = 200, 261, 512, 384
    A, b, sfb, scale2 = w4_inputs(M, N, K, 91)
    b_t, sfb_t = transposed(b, sfb, ldb, 92)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    C = buf[guard:guard + M * N].view(M, N)
    g.gemm_w4a16_t(to_dev_bf16(A), to_dev_u8(b_t), to_dev_u8(sfb_t), scale2, N, C)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + M * N:] == 7.0)
    check_close16(bits16(C), oracle.gemm_w4a16_t(A, b_t, sfb_t, scale2, N), K, amax(A),
                  wmax(b, sfb, scale2), what="guarded")


def test_w4a16_t_vocab_sized_odd_n_sampled(g):
    # an lm_head-like odd N (the page's motivating case) at ldb = align_up(N, 128)
    M, N, K = 4, 248077, 256
    ldb = align_up(N, 128)
    A, b, sfb, scale2 = w4_inputs(M, N, K, 111, 1.0)
    b_t, sfb_t = transposed(b, sfb, ldb, 112)
    got = run(g, A, b_t, sfb_t, scale2, N)
    cols = np.r_[0:300, N - 300:N, np.random.default_rng(5).integers(0, N, 400)]
    ref = oracle.gemm_w4a16_t(A, b_t[:, :], sfb_t, scale2, N)
    check_close16(got[:, cols], ref[:, cols], K, amax(A), wmax(b, sfb, scale2), what="vocab odd N")


def test_w4a16_t_qkvz_sampled(g):
    w = synth.W4A16["w4a16_qkvz"]
    A, b, sfb, scale2 = synth.w4a16_inputs(w)
    b_t, sfb_t = transposed(b, sfb, w.N, 121)
    got = run(g, A, b_t, sfb_t, scale2, w.N)
    rows = sample_rows(w.M, n_random=32, seed=11)
    ref = oracle.gemm_w4a16_t(A, b_t, sfb_t, scale2, w.N, rows=rows)
    stats = check_close16(got[rows], ref, w.K, amax(A), wmax(b, sfb, scale2), what="w4a16_t qkvz")
    assert stats["frac_exact"] > 0.9, stats


def test_w4a16_t_rejects_bad_stride(g):
    A = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    b_t = torch.zeros((128, 264), dtype=torch.uint8, device="cuda")   # ldb 264: not a multiple of 16
    s_t = torch.zeros((16, 264), dtype=torch.uint8, device="cuda")
    with pytest.raises(g.GemmError):
        g.gemm_w4a16_t(A, b_t, s_t, 1.0, 260)
    b_t = torch.zeros((128, 256), dtype=torch.uint8, device="cuda")   # ldb < N
    s_t = torch.zeros((16, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(g.GemmError):
        g.gemm_w4a16_t(A, b_t, s_t, 1.0, 257)
