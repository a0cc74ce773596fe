"""Pins for the CPU oracle: each oracle function is checked against something
other than itself (brute-force FP64, closed forms, library casts, the layout
statement of the NVFP4 page, hand-derived fixtures).  CPU only."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# e2m1 values by code, from the format definition (OCP Microscaling spec:
# 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def bf16_bits_to_f64(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def test_bf16_rne_matches_torch_cast_on_strided_fp32_patterns():
    # every 251st fp32 bit pattern (covers every exponent, both signs, many
    # tie cases) plus hand-picked ties and specials
    pats = np.arange(0, 2**32, 251, dtype=np.uint64).astype(np.uint32)
    extra = np.array([0x3f808000, 0x3f818000, 0x3f80_7fff, 0x3f80_8001, 0x7f7f_ffff,
                      0x7f80_0000, 0xff80_0000, 0x0000_8000, 0x0001_8000, 0x8000_0000,
                      0x7fc0_0000, 0x7f80_0001, 0x0080_8000], dtype=np.uint32)
    pats = np.concatenate([pats, extra])
    x = pats.view(np.float32)
    got = oracle.f32_to_bf16_array(x)
    ref = torch_bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    # NaN stays NaN (exponent all ones, nonzero mantissa), sign kept
    g = got[nan]
    assert np.all((g & 0x7f80) == 0x7f80) and np.all((g & 0x007f) != 0)
    assert np.array_equal(g >> 15, (pats[nan] >> 31).astype(np.uint16))


def test_bf16_roundtrip_exact():
    bits = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    f = bf16_bits_to_f64(bits).astype(np.float32)
    back = oracle.f32_to_bf16_array(f)
    ok = ~np.isnan(f)
    assert np.array_equal(back[ok], bits[ok])


def test_f16_rne_from_f64_matches_numpy():
    rng = np.random.default_rng(7)
    # magnitudes spanning subnormals, normals, the overflow edge
    e = rng.uniform(-27, 17, size=400_000)
    x = np.sign(rng.standard_normal(e.size)) * np.exp2(e)
    # exact ties in the normal and subnormal ranges, and the overflow boundary
    ties = []
    for ex in range(-24, 16):
        q = 2.0 ** max(ex - 10, -24)
        base = 2.0 ** ex
        ties += [base + q / 2, base + 3 * q / 2, -(base + q / 2)]
    ties += [65504.0, 65519.99, 65520.0, 65536.0, 1e9, 2.0**-25, 2.0**-25 * 1.0000001,
             3 * 2.0**-26, 0.0, -0.0, np.inf, -np.inf]
    x = np.concatenate([x, np.array(ties)])
    got = oracle.f64_to_f16_array(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)
    nan = oracle.f64_to_f16(float("nan"))
    assert (nan & 0x7c00) == 0x7c00 and (nan & 0x3ff) != 0


def test_f16_decode_all_patterns():
    bits = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits[::7]])
    r = ref[::7]
    both_nan = np.isnan(got) & np.isnan(r)
    assert np.array_equal(got[~both_nan], r[~both_nan])


def test_e2m1_table():
    got = [oracle.e2m1_decode(c) for c in range(16)]
    assert got == E2M1_TABLE
    assert [np.signbit(v) for v in got] == [c >= 8 for c in range(16)]


def test_e4m3_decode_matches_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert nan.sum() == 2  # 0x7f and 0xff
    # the power-of-two scale bytes the inputs use
    for e, byte in synth.E4M3_POW2_BYTES.items():
        assert oracle.e4m3_decode(byte) == 2.0**e


# --------------------------------------------------------------------------
# scale-factor layout
# --------------------------------------------------------------------------

def test_sf_offset_golden_examples():
    with open(os.path.join(GOLDEN, "sf_layout_examples.txt")) as f:
        rows = [ln.split("#")[0].split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 8
    for r, j, l, rest_m, rest_k, off in ([int(v) for v in row] for row in rows):
        assert oracle.sf_offset(r, j, l, rest_m, rest_k) == off, (r, j, l)


@pytest.mark.parametrize("L,M,K", [(1, 128, 64), (1, 256, 512), (2, 384, 256)])
def test_sf_offset_matches_page_permute(L, M, K):
    """The page stores the logical [32,4,rest_m,4,rest_k,L] tensor so that
    permute(5,2,4,0,1,3) is contiguous [L,rest_m,rest_k,32,4,4]; build that
    with torch from a logical [L,M,K/16] grid and compare byte by byte."""
    rest_m, rest_k = M // 128, K // 64
    g = torch.Generator().manual_seed(5)
    logical = torch.randint(0, 256, (L, M, K // 16), generator=g, dtype=torch.int32).to(torch.uint8)
    # logical[l, tile*128 + i_m*32 + g_m, tile_k*4 + i_k] -> six-dim [g_m,i_m,tile,i_k,tile_k,l]
    six = logical.reshape(L, rest_m, 4, 32, rest_k, 4).permute(3, 2, 1, 5, 4, 0)
    assert tuple(six.shape) == (32, 4, rest_m, 4, rest_k, L)
    phys = six.permute(5, 2, 4, 0, 1, 3).contiguous().reshape(-1).numpy()
    lg = logical.numpy()
    for l in range(L):
        for r in range(M):
            offs = [oracle.sf_offset(r, j, l, rest_m, rest_k) for j in range(K // 16)]
            assert np.array_equal(phys[offs], lg[l, r]), (l, r)
    # the map is a bijection onto the buffer
    all_offs = {oracle.sf_offset(r, j, l, rest_m, rest_k)
                for l in range(L) for r in range(M) for j in range(K // 16)}
    assert all_offs == set(range(L * M * K // 16))


# --------------------------------------------------------------------------
# BF16 GEMM, scaled-acc and router
# --------------------------------------------------------------------------

def _rand_bf16(shape, seed, sigma=1.0):
    return synth.bf16_normal(shape, sigma, seed)


@pytest.mark.parametrize("M,N,K", [(7, 5, 33), (16, 24, 64), (3, 40, 257)])
def test_router_within_higham_bound_of_fp64(M, N, K):
    A, B = _rand_bf16((M, K), 1), _rand_bf16((N, K), 2)
    a, b = bf16_bits_to_f64(A), bf16_bits_to_f64(B)
    exact = a @ b.T
    bound = (K - 1) * 2.0**-24 * (np.abs(a) @ np.abs(b).T) + 1e-300
    got = oracle.gemm_router(A, B).astype(np.float64)
    assert np.all(np.abs(got - exact) <= bound)


def test_router_rejects_transposed_operand_mistake():
    # a non-square case where A @ B (wrong) and A @ B^T differ grossly
    M, N, K = 4, 6, 6
    A, B = _rand_bf16((M, K), 3), _rand_bf16((N, K), 4)
    a, b = bf16_bits_to_f64(A), bf16_bits_to_f64(B)
    got = oracle.gemm_router(A, B).astype(np.float64)
    assert np.allclose(got, a @ b.T, rtol=1e-5, atol=1e-5)
    assert not np.allclose(got, a @ b, rtol=1e-2, atol=1e-2)


def test_router_strict_order_fma_and_subnormal_case():
    with open(os.path.join(GOLDEN, "router_fma_case.txt")) as f:
        vals = {ln.split()[0]: [int(v, 16) for v in ln.split()[1:]]
                for ln in f if ln.strip() and not ln.startswith("#")}
    A = np.array([vals["a_bf16"]], dtype=np.uint16)
    B = np.array([vals["b_bf16"]], dtype=np.uint16)
    got = oracle.gemm_router(A, B).view(np.uint32)
    assert got[0, 0] == vals["c_f32"][0]


def test_router_zero_rows_give_positive_zero():
    A = np.zeros((2, 8), dtype=np.uint16)
    A[1] = 0x8000  # -0.0 everywhere
    B = _rand_bf16((3, 8), 9)
    got = oracle.gemm_router(A, B).view(np.uint32)
    assert np.all(got == 0)


def test_router_is_sequential_fp32_sum():
    # Catastrophic-cancellation case with a known sequential answer:
    # 2^24 + 1 - 2^24 in fp32, in k order, is 0 (the +1 is absorbed).
    A = np.array([[0x4b80, 0x3f80, 0xcb80]], dtype=np.uint16)  # 2^24, 1, -2^24
    B = np.array([[0x3f80, 0x3f80, 0x3f80]], dtype=np.uint16)
    assert oracle.gemm_router(A, B)[0, 0] == 0.0
    # reversed order keeps the 1: -2^24 + 1 = -16777215 exactly, + 2^24 = 1
    A2 = A[:, ::-1].copy()
    B2 = B[:, ::-1].copy()
    assert oracle.gemm_router(A2, B2)[0, 0] == 1.0


@pytest.mark.parametrize("M,N,K", [(9, 17, 40), (32, 8, 128)])
def test_bf16_gemm_is_rne_of_router_sum_and_close_to_exact(M, N, K):
    A, B = _rand_bf16((M, K), 11), _rand_bf16((N, K), 12)
    C = oracle.gemm_bf16_nt(A, B)
    R = oracle.gemm_router(A, B)
    assert np.array_equal(C, torch_bf16_bits(R))
    a, b = bf16_bits_to_f64(A), bf16_bits_to_f64(B)
    exact = a @ b.T
    c = bf16_bits_to_f64(C)
    seq = (K - 1) * 2.0**-24 * (np.abs(a) @ np.abs(b).T)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact) + seq, 1e-30))) - 8)
    assert np.all(np.abs(c - exact) <= seq + half_ulp)


def test_bf16_gemm_identity_and_permutation():
    K = 64
    A = _rand_bf16((24, K), 21)
    eye = np.zeros((K, K), dtype=np.uint16)
    eye[np.arange(K), np.arange(K)] = 0x3f80
    assert np.array_equal(oracle.gemm_bf16_nt(A, eye), A)
    perm = np.random.default_rng(3).permutation(K)
    P = np.zeros((K, K), dtype=np.uint16)
    P[np.arange(K), perm] = 0x3f80  # row n of B picks column perm[n] of A
    assert np.array_equal(oracle.gemm_bf16_nt(A, P), A[:, perm])


def test_bf16_gemm_exact_integers():
    M, N, K = 20, 30, 256
    A = synth.bf16_small_ints((M, K), -3, 3, 31)
    B = synth.bf16_small_ints((N, K), -3, 3, 32)
    ai = bf16_bits_to_f64(A).astype(np.int64)
    bi = bf16_bits_to_f64(B).astype(np.int64)
    exact = ai @ bi.T
    assert np.abs(exact).max() < 2**24
    assert np.array_equal(oracle.gemm_bf16_nt(A, B), torch_bf16_bits(exact.astype(np.float32)))
    assert np.array_equal(oracle.gemm_router(A, B), exact.astype(np.float32))


@pytest.mark.parametrize("scale", [0.5, 2.0, -0.37])
def test_scaled_acc_fused_equals_unfused_and_closed_form(scale):
    M, N, K = 12, 40, 48
    A, B = _rand_bf16((M, K), 41), _rand_bf16((N, K), 42)
    out0 = _rand_bf16((M, N), 43)
    fused = oracle.gemm_bf16_nt_scaled_acc(A, B, out0, scale)
    d = oracle.gemm_bf16_nt(A, B)
    unfused = oracle.bf16_scaled_add(out0, d, scale)
    assert np.array_equal(fused, unfused)
    # closed form with library casts: bf16(fp32(out) + fp32(scale*fp32(d)))
    o32 = bf16_bits_to_f64(out0).astype(np.float32)
    d32 = bf16_bits_to_f64(d).astype(np.float32)
    ref = torch_bf16_bits(o32 + np.float32(scale) * d32)
    assert np.array_equal(fused, ref)


def test_scaled_acc_row_selection():
    M, N, K = 10, 16, 32
    A, B = _rand_bf16((M, K), 51), _rand_bf16((N, K), 52)
    out0 = _rand_bf16((M, N), 53)
    full = oracle.gemm_bf16_nt_scaled_acc(A, B, out0, 0.5)
    rows = [9, 0, 4]
    part = oracle.gemm_bf16_nt_scaled_acc(A, B, out0[rows], 0.5, rows=rows)
    assert np.array_equal(part, full[rows])
    assert np.array_equal(oracle.gemm_bf16_nt(A, B, rows=rows), oracle.gemm_bf16_nt(A, B)[rows])


# --------------------------------------------------------------------------
# NVFP4 block-scaled GEMM
# --------------------------------------------------------------------------

def nvfp4_reference_f64(a, b, sfa, sfb, L, M, N, K):
    """Independent FP64 evaluation: literal e2m1 table, torch's e4m3 cast and
    the page's permute to recover the logical scale grid."""
    tab = np.array(E2M1_TABLE)
    def dequant_codes(x, rows):
        x = x.reshape(L, rows, K // 2)
        codes = np.empty((L, rows, K), dtype=np.uint8)
        codes[..., 0::2] = x & 0x0F   # reading: even k in the low nibble
        codes[..., 1::2] = x >> 4
        return tab[codes]
    def logical_scales(sf, rows):
        phys = torch.from_numpy(sf.reshape(L, rows // 128, K // 64, 32, 4, 4).copy())
        # physical [l, tile, tile_k, g, i_m, i_k] -> logical [l, tile, i_m, g, tile_k, i_k]
        lg = phys.permute(0, 1, 4, 3, 2, 5).reshape(L, rows, K // 16)
        return lg.contiguous().view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    av = dequant_codes(a, M) * np.repeat(logical_scales(sfa, M), 16, axis=2)
    bv = dequant_codes(b, N) * np.repeat(logical_scales(sfb, N), 16, axis=2)
    return np.einsum("lmk,lnk->lmn", av, bv)


@pytest.mark.parametrize("L,M,N,K", [(1, 128, 128, 64), (1, 256, 128, 256), (2, 128, 256, 128)])
def test_nvfp4_matches_independent_fp64(L, M, N, K):
    w = synth.Nvfp4("t", L, M, N, K, 77)
    a, b, sfa, sfb = synth.nvfp4_inputs(w)
    exact = nvfp4_reference_f64(a, b, sfa, sfb, L, M, N, K)
    got = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K)
    assert np.array_equal(got, exact.reshape(L * M, N).astype(np.float16).view(np.uint16))


def test_nvfp4_identity_gives_dequantised_a():
    L, M, N, K = 1, 128, 128, 128
    w = synth.Nvfp4("t", L, M, N, K, 78)
    a, _, sfa, _ = synth.nvfp4_inputs(w)
    # b = identity: code 0x2 (1.0) at k == n, zero elsewhere; unit scales (0x38)
    b = np.zeros((L, N, K // 2), dtype=np.uint8)
    for n in range(N):
        b[0, n, n // 2] |= (0x2 << (4 * (n % 2)))
    sfb = np.full(L * N * K // 16, 0x38, dtype=np.uint8)
    got = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K)
    deq = nvfp4_reference_f64(a, np.broadcast_to(b, b.shape).copy(), sfa, sfb, L, M, N, K)
    assert np.array_equal(got, deq.reshape(M, N).astype(np.float16).view(np.uint16))
    # and directly: c[m, n] = e2m1(a[m, n]) * sfa(m, n/16)
    m, n = 77, 33
    code = (a[0, m, n // 2] >> (4 * (n % 2))) & 0xF
    s = oracle.e4m3_decode(sfa[oracle.sf_offset(m, n // 16, 0, M // 128, K // 64)])
    assert oracle.f16_to_f64(int(got[m, n])) == E2M1_TABLE[code] * s


def test_nvfp4_one_hot_scale_changes_one_block():
    L, M, N, K = 1, 128, 128, 128
    w = synth.Nvfp4("t", L, M, N, K, 79)
    a, b, sfa, sfb = synth.nvfp4_inputs(w)
    sfa[:] = 0x38
    sfb[:] = 0x38
    base = nvfp4_reference_f64(a, b, sfa, sfb, L, M, N, K)[0]
    r, j = 70, 5                      # row 70, k block 5 (k = 80..95)
    sfa2 = sfa.copy()
    sfa2[oracle.sf_offset(r, j, 0, 1, K // 64)] = 0x40   # scale 2.0
    got = oracle.gemm_nvfp4_bs(a, b, sfa2, sfb, L, M, N, K).view(np.float16).astype(np.float64)
    tab = np.array(E2M1_TABLE)
    def codes(x, row):
        c = np.empty(K, dtype=np.uint8)
        c[0::2] = x[0, row] & 0xF
        c[1::2] = x[0, row] >> 4
        return tab[c]
    block = sum(codes(a, r)[k] * np.array([codes(b, n)[k] for n in range(N)]) for k in range(80, 96))
    expect = base.copy()
    expect[r] += block
    assert np.array_equal(got, expect.astype(np.float16).astype(np.float64))
    others = np.delete(np.arange(M), r)
    assert np.array_equal(got[others], base[others].astype(np.float16).astype(np.float64))


def test_nvfp4_row_selection_batched():
    L, M, N, K = 2, 128, 128, 64
    w = synth.Nvfp4("t", L, M, N, K, 80)
    a, b, sfa, sfb = synth.nvfp4_inputs(w)
    full = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K)
    rows = [200, 3, 255, 128]
    part = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K, rows=rows)
    assert np.array_equal(part, full[rows])


def test_nvfp4_fp16_overflow_to_inf():
    L, M, N, K = 1, 128, 128, 64
    a = np.full((L, M, K // 2), 0x77, dtype=np.uint8)   # every code 6.0
    b = np.full((L, N, K // 2), 0x77, dtype=np.uint8)
    sf = np.full(L * M * K // 16, 0x48, dtype=np.uint8)  # scale 4.0
    got = oracle.gemm_nvfp4_bs(a, b, sf, sf, L, M, N, K)
    # 64 * (6*4)^2 = 36864 (finite); with scale 4 on both: exact sum 36864 -> fp16 36864
    assert oracle.f16_to_f64(int(got[0, 0])) == 36864.0
    a2 = np.full((L, M, K // 2), 0x77, dtype=np.uint8)
    sf2 = np.full(L * M * K // 16, 0x50, dtype=np.uint8)  # scale 8.0 -> 64*48*48 = 147456 > 65504
    got2 = oracle.gemm_nvfp4_bs(a2, b, sf2, sf2, L, M, N, K)
    assert got2[0, 0] == 0x7c00


# --------------------------------------------------------------------------
# W4A16: BF16 activations x NVFP4 weights
# --------------------------------------------------------------------------

def _w4_one_weight(code: int, scale_byte: int, scale2: float) -> int:
    """C[0,0] of a 1 x 1 x 16 W4A16 GEMM whose only nonzero product is
    A[0,0] = 1 times weight (code, scale): the dequantised weight itself."""
    A = np.zeros((1, 16), dtype=np.uint16)
    A[0, 0] = 0x3F80
    b = np.zeros((1, 8), dtype=np.uint8)
    b[0, 0] = code & 0xF           # k = 0: low nibble
    sfb = np.full((1, 1), scale_byte, dtype=np.uint8)
    return int(oracle.gemm_w4a16(A, b, sfb, scale2)[0, 0])


def test_w4a16_dequant_golden_examples():
    with open(os.path.join(GOLDEN, "w4a16_dequant_examples.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 8
    for code, sb, s2, want in rows:
        scale2 = float(np.array([int(s2, 16)], dtype=np.uint32).view(np.float32)[0])
        got = _w4_one_weight(int(code, 16), int(sb, 16), scale2)
        assert got == int(want, 16), (code, sb, s2, hex(got), want)


def test_w4a16_nibble_order_and_scale_groups():
    # row 0 of b: k=0 -> 1.0 (code 2, low nibble of byte 0), k=1 -> 2.0 (code 4,
    # high nibble), k=16 -> 1.0 (code 2) in scale group 1 (scale 2.0); group 0
    # has scale 1.0.  One-hot rows of A pick out single weights.
    K = 32
    b = np.zeros((1, K // 2), dtype=np.uint8)
    b[0, 0] = 0x42
    b[0, 8] = 0x02
    sfb = np.array([[0x38, 0x40]], dtype=np.uint8)
    A = np.zeros((3, K), dtype=np.uint16)
    A[0, 0] = A[1, 1] = A[2, 16] = 0x3F80
    got = bf16_bits_to_f64(oracle.gemm_w4a16(A, b, sfb, 1.0)[:, 0])
    assert got.tolist() == [1.0, 2.0, 2.0]


@pytest.mark.parametrize("M,N,K,e2", [(7, 24, 64, 0), (33, 16, 160, -3), (5, 40, 32, 2)])
def test_w4a16_exact_integers_match_integer_matmul(M, N, K, e2):
    # scales 2.0 (0x40) make every e2m1 value times the scale an integer in
    # {0, 1, 2, 3, 4, 6, 8, 12} up to sign; scale2 = 2^e2 keeps them exact, and
    # small-integer activations keep every FP32 partial sum exact.
    rng = np.random.default_rng(M * N + K)
    A = synth.bf16_small_ints((M, K), -4, 4, M + K)
    b = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sfb = np.full((N, K // 16), 0x40, dtype=np.uint8)
    tab = np.array(E2M1_TABLE)
    codes = np.empty((N, K), dtype=np.uint8)
    codes[:, 0::2] = b & 0xF
    codes[:, 1::2] = b >> 4
    w = (tab[codes] * 2.0 * 2.0**e2)
    exact = bf16_bits_to_f64(A) @ w.T
    got = oracle.gemm_w4a16(A, b, sfb, 2.0**e2)
    assert np.array_equal(got, torch_bf16_bits(exact.astype(np.float32)))


def _torch_block_scaled(b, sfb, N, K):
    """e2m1 * e4m3 weights from the format tables and torch's e4m3 cast (float32, exact)."""
    tab = torch.tensor(E2M1_TABLE, dtype=torch.float32)
    codes = torch.empty((N, K), dtype=torch.long)
    bt = torch.from_numpy(b.astype(np.int64))
    codes[:, 0::2] = bt & 0xF
    codes[:, 1::2] = bt >> 4
    sc = torch.from_numpy(sfb.copy()).view(torch.float8_e4m3fn).to(torch.float32)
    return tab[codes] * sc.repeat_interleave(16, dim=1)


def test_w4a16_equals_bf16_gemm_on_torch_dequantised_weights():
    # the block-scaled weights built by torch are exact in bf16; with
    # scale2 = 1 the W4A16 oracle is the pinned BF16 oracle GEMM on them, and
    # with any scale2 it is the pinned strict FP32 sum times scale2, rounded
    # by torch's float32 multiply and bfloat16 cast
    w = synth.W4a16("t", 37, 48, 96, 0.37, 91)
    A, b, sfb, scale2 = synth.w4a16_inputs(w)
    q = _torch_block_scaled(b, sfb, w.N, w.K)
    W = q.to(torch.bfloat16)
    assert torch.equal(W.to(torch.float32), q)  # exact in bf16
    W = W.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.gemm_w4a16(A, b, sfb, 1.0), oracle.gemm_bf16_nt(A, W))
    acc = torch.from_numpy(oracle.gemm_router(A, W))
    want = (acc * torch.tensor(scale2, dtype=torch.float32)).to(torch.bfloat16)
    assert np.array_equal(oracle.gemm_w4a16(A, b, sfb, scale2),
                          want.view(torch.int16).numpy().view(np.uint16))


def test_w4a16_within_fp32_bound_of_fp64():
    w = synth.W4a16("t", 19, 40, 256, 0.0123, 92)
    A, b, sfb, scale2 = synth.w4a16_inputs(w)
    tab = np.array(E2M1_TABLE)
    codes = np.empty((w.N, w.K), dtype=np.uint8)
    codes[:, 0::2] = b & 0xF
    codes[:, 1::2] = b >> 4
    sc = torch.from_numpy(sfb.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    wv = tab[codes] * np.repeat(sc, 16, axis=1) * scale2
    a = bf16_bits_to_f64(A)
    exact = a @ wv.T
    got = bf16_bits_to_f64(oracle.gemm_w4a16(A, b, sfb, scale2))
    # FP32 accumulation (K * 2^-24), the FP32 scale product and the output rounding
    bound = (w.K + 1) * 2.0**-24 * (np.abs(a) @ np.abs(wv).T) + 2.0**-8 * np.abs(exact)
    assert np.all(np.abs(got - exact) <= bound + 1e-30)
    # and a wrong nibble order would break it
    codes_sw = codes.copy()
    codes_sw[:, 0::2], codes_sw[:, 1::2] = codes[:, 1::2], codes[:, 0::2]
    wrong = a @ (tab[codes_sw] * np.repeat(sc, 16, axis=1) * scale2).T
    assert not np.all(np.abs(got - wrong) <= bound + 1e-30)


def test_w4a16_row_selection():
    w = synth.W4a16("t", 21, 16, 64, 0.5, 93)
    A, b, sfb, scale2 = synth.w4a16_inputs(w)
    full = oracle.gemm_w4a16(A, b, sfb, scale2)
    rows = [20, 0, 7]
    assert np.array_equal(oracle.gemm_w4a16(A, b, sfb, scale2, rows=rows), full[rows])


# --------------------------------------------------------------------------
# W4A16 with the transposed weight layout
# --------------------------------------------------------------------------

def test_w4a16_t_layout_golden_examples():
    with open(os.path.join(GOLDEN, "w4a16_t_layout_examples.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 5
    for K, N, ldb, k, n, boff, nib, code, soff, sb, want in rows:
        K, N, ldb, k, n, boff, soff = map(int, (K, N, ldb, k, n, boff, soff))
        b_t = np.zeros((K // 2, ldb), dtype=np.uint8)
        sfb_t = np.full((K // 16, ldb), 0x38, dtype=np.uint8)
        c = int(code, 16)
        b_t.reshape(-1)[boff] = c if nib == "lo" else c << 4
        sfb_t.reshape(-1)[soff] = int(sb, 16)
        A = np.zeros((1, K), dtype=np.uint16)
        A[0, k] = 0x3F80
        got = oracle.gemm_w4a16_t(A, b_t, sfb_t, 1.0, N)
        assert int(got[0, n]) == int(want, 16), (k, n, hex(int(got[0, n])), want)
        others = np.delete(got[0], n)
        assert np.all((others & 0x7FFF) == 0), others   # no other column sees the weight


@pytest.mark.parametrize("M,N,K,ldb", [(9, 32, 64, 32), (13, 37, 96, 128), (6, 129, 32, 256)])
def test_w4a16_t_equals_row_layout_under_transpose(M, N, K, ldb):
    # the transposed layout is the [N][K/2] byte matrix (and the [N][K/16]
    # scale matrix) transposed, rows padded to ldb bytes with junk that must
    # never be read
    rng = np.random.default_rng(M + N + K)
    w = synth.W4a16("t", M, N, K, 0.75, 95 + N)
    A, b, sfb, scale2 = synth.w4a16_inputs(w)
    b_t = rng.integers(0, 256, (K // 2, ldb), dtype=np.uint8)
    sfb_t = rng.integers(0, 256, (K // 16, ldb), dtype=np.uint8)
    b_t[:, :N] = b.T
    sfb_t[:, :N] = sfb.T
    want = oracle.gemm_w4a16(A, b, sfb, scale2)
    assert np.array_equal(oracle.gemm_w4a16_t(A, b_t, sfb_t, scale2, N), want)
    # a layout read along the wrong axis would not agree
    if N == K // 2 and ldb == N:
        assert not np.array_equal(oracle.gemm_w4a16_t(A, b, sfb_t, scale2, N), want)


def test_w4a16_t_rejects_short_stride():
    A = np.zeros((1, 32), dtype=np.uint16)
    with pytest.raises(AssertionError):
        oracle.gemm_w4a16_t(A, np.zeros((16, 4), np.uint8), np.zeros((2, 4), np.uint8), 1.0, 5)
