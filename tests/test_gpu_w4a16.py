"""GPU parity of the W4A16 GEMM (BF16 activations x NVFP4 weights) against the
CPU oracle, through the C ABI."""
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


def run(g, A, b, sfb, scale2):
    return bits16(g.gemm_w4a16(to_dev_bf16(A), to_dev_u8(b), to_dev_u8(sfb), scale2))


def wmax(b, sfb, scale2):
    """Largest |dequantised weight| (for the tolerance rule)."""
    tab = np.abs(np.array(E2M1))
    hi = np.maximum(tab[b & 0xF], tab[b >> 4]).reshape(b.shape[0], -1, 8).max(axis=2)
    sc = torch.from_numpy(sfb.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return float((hi * sc).max() * abs(scale2))


def amax(x):
    return float(np.abs(bf16_val(x)).max())


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 256),     # one tile
    (300, 520, 768),     # ragged M and N; three pairs of K blocks
    (1, 8, 256),         # degenerate
    (129, 264, 512),     # one row / 8 columns past a tile
    (17, 1000, 2304),    # many stages, N not a multiple of 256
    (640, 768, 256),     # exact multiples
    (1100, 1032, 768),   # five M blocks: the last work item's second tile lies past M
])
def test_w4a16_ragged(g, M, N, K):
    w = synth.W4a16("t", M, N, K, 0.37, 300 + M)
    A, b, sfb, scale2 = synth.w4a16_inputs(w)
    got = run(g, A, b, sfb, scale2)
    ref = oracle.gemm_w4a16(A, b, sfb, scale2)
    check_close16(got, ref, K, amax(A), wmax(b, sfb, scale2), what=f"w4a16 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,e2", [(384, 520, 512, -2), (256, 256, 2048, 0), (77, 136, 256, 1)])
def test_w4a16_exact_integers_bitexact(g, M, N, K, e2):
    # block scales 2.0 and scale2 = 2^e2 make every weight a small integer
    # times 2^e2; small-integer activations keep every FP32 sum exact
    A = synth.bf16_small_ints((M, K), -3, 3, 21 + K)
    b = synth.uniform_bytes(N * K // 2, 22 + K).reshape(N, K // 2)
    sfb = np.full((N, K // 16), 0x40, dtype=np.uint8)
    got = run(g, A, b, sfb, 2.0**e2)
    check_bitexact16(got, oracle.gemm_w4a16(A, b, sfb, 2.0**e2), f"w4a16 exact {M}x{N}x{K}")


def test_w4a16_identity_reads_back_every_weight(g):
    # A = I (K x K): C[m, n] = w[n, m], one product per output, so the
    # dequantised weights come back bit for bit (nibble order, scale groups,
    # rounding of the per-tensor scale, subnormal and varied e4m3 scales)
    K, N = 256, 264
    A = np.zeros((K, K), dtype=np.uint16)
    A[np.arange(K), np.arange(K)] = 0x3F80
    b = synth.uniform_bytes(N * K // 2, 31).reshape(N, K // 2)
    sfb = synth.e4m3_range_bytes(N * K // 16, 32, 0x01, 0x7E).reshape(N, K // 16)
    for scale2 in (1.0, 0.0123, -3.7):
        check_bitexact16(run(g, A, b, sfb, scale2), oracle.gemm_w4a16(A, b, sfb, scale2),
                         f"identity scale2={scale2}")


def test_w4a16_equals_bf16_gemm_of_dequantised_weights(g):
    # the block-scaled weights are exact in bf16, and the kernel runs the
    # dense GEMM's tiles and MMA sequence on them: with scale2 = 1 the result
    # is bit-equal to gemm_bf16_nt on the weights dequantised on the host
    w = synth.W4a16("t", 520, 776, 512, 1.0, 41)
    A, b, sfb, _ = synth.w4a16_inputs(w)
    tab = torch.tensor(E2M1, dtype=torch.float32)
    codes = torch.empty((w.N, w.K), dtype=torch.long)
    bt = torch.from_numpy(b.astype(np.int64))
    codes[:, 0::2] = bt & 0xF
    codes[:, 1::2] = bt >> 4
    sc = torch.from_numpy(sfb.copy()).view(torch.float8_e4m3fn).to(torch.float32)
    W = (tab[codes] * sc.repeat_interleave(16, dim=1)).to(torch.bfloat16)
    W = W.view(torch.int16).numpy().view(np.uint16)
    dense = bits16(g.gemm_bf16_nt(to_dev_bf16(A), to_dev_bf16(W)))
    check_bitexact16(run(g, A, b, sfb, 1.0), dense, "w4a16 vs dense on dequantised weights")


def test_w4a16_no_write_outside_c(g):
    M, N, K = 200, 264, 512
    w = synth.W4a16("t", M, N, K, 0.5, 51)
    A, b, sfb, scale2 = synth.w4a16_inputs(w)
    guard = 4096
    buf = torch.full((guard + M * N + guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    C = buf[guard:guard + M * N].view(M, N)
    g.gemm_w4a16(to_dev_bf16(A), to_dev_u8(b), to_dev_u8(sfb), scale2, C)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + M * N:] == 7.0)
    check_close16(bits16(C), oracle.gemm_w4a16(A, b, sfb, scale2), K, amax(A),
                  wmax(b, sfb, scale2), what="guarded")


def test_w4a16_full_size_sampled(g):
    w = synth.W4A16["w4a16_qkvz"]
    A, b, sfb, scale2 = synth.w4a16_inputs(w)
    got = run(g, A, b, sfb, scale2)
    rows = sample_rows(w.M, n_random=48, seed=9)
    ref = oracle.gemm_w4a16(A, b, sfb, scale2, rows=rows)
    stats = check_close16(got[rows], ref, w.K, amax(A), wmax(b, sfb, scale2), what="w4a16 qkvz")
    assert stats["frac_exact"] > 0.9, stats


def _random_shapes(seed, count):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(1, 1200)), int(rng.integers(1, 200)) * 8, int(rng.integers(1, 10)) * 256)
            for _ in range(count)]


@pytest.mark.parametrize("M,N,K", _random_shapes(4242, 6))
def test_w4a16_random_shapes_exact_integers(g, M, N, K):
    # seeded ragged shapes; block scales 2^{-1..1}, integer activations and a
    # power-of-two per-tensor scale keep every sum exact: bit-exact
    rng = np.random.default_rng(M * 7 + N)
    A = synth.bf16_small_ints((M, K), -3, 3, M + K)
    b = synth.uniform_bytes(N * K // 2, N + K).reshape(N, K // 2)
    sfb = rng.choice(np.array([0x30, 0x38, 0x40], dtype=np.uint8), size=(N, K // 16))
    got = run(g, A, b, sfb, 0.5)
    check_bitexact16(got, oracle.gemm_w4a16(A, b, sfb, 0.5), f"w4a16 random {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(300, 520, 768), (1, 8, 256), (1016, 12288, 2048),
                                   (129, 264, 512)])
def test_w4a16_two_pass_equals_fused(g, M, N, K):
    # same tiles, K order and epilogue: bit-identical to the fused kernel,
    # and the workspace holds the exact converted weights
    w = synth.W4a16("t", M, N, K, 0.0123, 500 + M)
    A, b, sfb, scale2 = synth.w4a16_inputs(w)
    Ad, bd, sd = to_dev_bf16(A), to_dev_u8(b), to_dev_u8(sfb)
    ws = torch.empty(g.gemm_w4a16_ws_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    two = bits16(g.gemm_w4a16_ws(Ad, bd, sd, scale2, ws))
    fused = bits16(g.gemm_w4a16(Ad, bd, sd, scale2))
    check_bitexact16(two, fused, f"two-pass vs fused {M}x{N}x{K}")
    if M <= 512:
        check_close16(two, oracle.gemm_w4a16(A, b, sfb, scale2), K, amax(A),
                      wmax(b, sfb, scale2), what="two-pass vs oracle")
    # the converted weights: one-hot rows of A read them back through the oracle
    W = ws.view(torch.int16).view(N, K).cpu().numpy().view(np.uint16)
    eye = np.zeros((K, K), dtype=np.uint16)
    eye[np.arange(K), np.arange(K)] = 0x3F80
    ref = oracle.gemm_w4a16(eye, b[:8], sfb[:8], 1.0)       # [K][8]: weights of rows 0..7
    check_bitexact16(W[:8].T.copy(), ref, "converted weights")


def test_w4a16_two_pass_rejects_a_small_workspace(g):
    A = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((256, 128), dtype=torch.uint8, device="cuda")
    s = torch.zeros((256, 16), dtype=torch.uint8, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.GemmError):
        g.gemm_w4a16_ws(A, b, s, 1.0, ws)
