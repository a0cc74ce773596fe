"""GPU parity where the result is not finite: a non-finite output passes
only where the oracle has the same one.

* NVFP4 (FP16 output): rows whose exact sums sit on the FP16 overflow edge
  (65504 stays finite; 65520 is the midpoint to the next binade and rounds
  to +inf under ties-to-even), far past it (+inf and -inf), and a row whose
  huge terms cancel exactly.  Through gemm_nvfp4_bs and through the split-K
  path, whose FP32 chunks are finite and overflow only in the FP16 reduce.
* Fused scaled-acc: `out` holding +inf, -inf and NaN, and a delta that
  overflows BF16 (every product of the row has the same sign, so the FP32
  sum is +inf in any summation order); the unfused GPU pair must agree bit
  for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import (bf16_val, bits16, check_bitexact16, check_close16, check_scaled_acc,
                    f16_val, to_dev_bf16, to_dev_u8)

pytestmark = pytest.mark.gpu

E2M1 = {0.0: 0x0, 0.5: 0x1, 1.0: 0x2, 1.5: 0x3, 2.0: 0x4, 3.0: 0x5, 4.0: 0x6, 6.0: 0x7}
NEG = 0x8
SCALE_ONE, SCALE_32 = 0x38, 0x60   # e4m3 1.0 and 2^5


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_tcgen05_gb300 as lib
    yield lib
    assert lib.gemm_get_device_status() == 0


def _pack(codes: np.ndarray) -> np.ndarray:
    """[rows, K] 4-bit codes -> [rows, K/2] bytes, element 2j in the low nibble."""
    c = codes.astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _edge_block(total_codes: list) -> np.ndarray:
    out = np.zeros(16, dtype=np.uint8)
    for i, v in enumerate(total_codes):
        out[i] = v
    return out


def nvfp4_edge_inputs(M=256, N=256, K=512, seed=301):
    """a, b, sfa, sfb (L = 1) whose first rows hit the FP16 overflow cases
    (K >= 512; codes past the first 512 of those rows are zero).

    b is code 1.0 everywhere with unit scales, so C[r, n] is row r's sum of
    dequantised a.  Rows 0..4 use scale 2^5 in every block:
      31 full blocks of 4.0 codes give 31 * 16 * 4 * 32 = 63488; block 31
      adds ten 6.0 codes, one 3.0 and one 0.5 (63.5 * 32 = 2032) -> 65520,
      or ten 6.0 and one 3.0 (63 * 32 = 2016) -> 65504.
    """
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(M, K), dtype=np.uint8)   # random rows elsewhere
    rest_k = K // 64
    sfa = synth.pow2_scale_bytes(M * K // 16, seed + 1)
    four = np.full(16, E2M1[4.0], dtype=np.uint8)
    tail_65520 = _edge_block([E2M1[6.0]] * 10 + [E2M1[3.0], E2M1[0.5]])
    tail_65504 = _edge_block([E2M1[6.0]] * 10 + [E2M1[3.0]])
    six = np.full(16, E2M1[6.0], dtype=np.uint8)
    rows = {
        0: np.concatenate([four] * 31 + [tail_65520]),                 # 65520 -> +inf
        1: np.concatenate([four] * 31 + [tail_65504]),                 # 65504 (max finite)
        2: np.concatenate([four | NEG] * 31 + [tail_65520 | NEG * (tail_65520 != 0)]),  # -65520 -> -inf
        3: np.concatenate([six] * 32),                                 # 98304 -> +inf
        4: np.concatenate([six] * 16 + [six | NEG] * 16),              # exactly 0
    }
    for r, c in rows.items():
        codes[r] = np.concatenate([c, np.zeros(K - c.size, dtype=np.uint8)])
        for j in range(K // 16):
            sfa[oracle.sf_offset(r, j, 0, M // 128, rest_k)] = SCALE_32
    a = _pack(codes).reshape(1, M, K // 2)
    b = _pack(np.full((N, K), E2M1[1.0], dtype=np.uint8)).reshape(1, N, K // 2)
    sfb = np.full(N * K // 16, SCALE_ONE, dtype=np.uint8)
    return a, b, sfa, sfb


def _oracle_edge(a, b, sfa, sfb, M, N, K):
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, 1, M, N, K).reshape(M, N)
    v = f16_val(ref)
    # the inputs exercise what they are meant to
    assert np.all(v[0] == np.inf) and np.all(v[3] == np.inf) and np.all(v[2] == -np.inf)
    assert np.all(v[1] == 65504.0) and np.all(v[4] == 0.0)
    return ref


def test_nvfp4_fp16_overflow(g):
    M, N, K = 256, 256, 512
    a, b, sfa, sfb = nvfp4_edge_inputs(M, N, K)
    ref = _oracle_edge(a, b, sfa, sfb, M, N, K)
    c = g.gemm_nvfp4_bs(to_dev_u8(a), to_dev_u8(b), to_dev_u8(sfa), to_dev_u8(sfb), 1, M, N, K)
    got = bits16(c).reshape(M, N)
    check_bitexact16(got[:5], ref[:5], "nvfp4 overflow rows", zero_sign=False)
    check_close16(got, ref, K, 6.0 * 32, 1.0, "f16", "nvfp4 with overflow rows")


@pytest.mark.parametrize("K,k_splits", [(512, 2), (1024, 4)])
def test_nvfp4_splitk_fp16_overflow(g, K, k_splits):
    # each FP32 chunk is finite; only the ordered FP16 reduce overflows
    M, N = 128, 256
    a, b, sfa, sfb = nvfp4_edge_inputs(M, N, K, seed=302)
    ref = _oracle_edge(a, b, sfa, sfb, M, N, K)
    c = g.gemm_nvfp4_bs_splitk(to_dev_u8(a), to_dev_u8(b), to_dev_u8(sfa), to_dev_u8(sfb),
                               M, N, K, k_splits)
    got = bits16(c).reshape(M, N)
    check_bitexact16(got[:5], ref[:5], f"nvfp4 split-K {k_splits} overflow rows")
    check_close16(got, ref, K, 6.0 * 32, 1.0, "f16", f"nvfp4 split-K {k_splits} with overflow rows")


BF16_INF, BF16_NINF, BF16_NAN = 0x7F80, 0xFF80, 0x7FC0


@pytest.mark.parametrize("M,N,K", [(256, 512, 16), (300, 264, 64), (128, 256, 2048)])
def test_scaled_acc_nonfinite_out_and_delta(g, M, N, K):
    scale = 2.0
    A = synth.bf16_normal((M, K), 1.0, 311 + K)
    B = synth.bf16_normal((N, K), 0.01, 312 + K)
    # row 5 of A and column 7 of B: 2^64 everywhere -> every product of
    # output (5, 7) is 2^128 > FP32 max, so the delta there is +inf
    big = np.uint16(0x5F80)   # bf16 2^64
    A[5, :] = big
    B[7, :] = big
    out0 = synth.bf16_normal((M, N), 1.0, 313 + K)
    rng = np.random.default_rng(314)
    idx = rng.choice(M * N, size=96, replace=False)
    flat = out0.reshape(-1)
    flat[idx[:32]] = BF16_INF
    flat[idx[32:64]] = BF16_NINF
    flat[idx[64:]] = BF16_NAN
    out0[5, 7] = 0x3F80        # finite out where the delta is +inf
    out0[5, 8] = BF16_NINF     # -inf + 2*(finite)
    out0[6, 7] = BF16_INF
    ref = oracle.gemm_bf16_nt_scaled_acc(A, B, out0, scale)
    refv = bf16_val(ref)
    assert np.isnan(refv).sum() >= 32 and np.isinf(refv).sum() >= 64
    assert refv[5, 7] == np.inf
    Ad, Bd = to_dev_bf16(A), to_dev_bf16(B)
    fused = to_dev_bf16(out0)
    g.gemm_bf16_nt_scaled_acc(Ad, Bd, fused, scale)
    got = bits16(fused)
    d_ref = oracle.gemm_bf16_nt(A, B)
    amax_a = float(np.abs(bf16_val(np.delete(A, 5, axis=0))).max())
    amax_b = float(np.abs(bf16_val(np.delete(B, 7, axis=0))).max())
    finite_rows = np.array([r for r in range(M) if r != 5])
    check_scaled_acc(got[finite_rows], ref[finite_rows], d_ref[finite_rows], scale, K, amax_a,
                     amax_b, f"scaled-acc non-finite out {M}x{N}x{K}")
    # row 5: delta +inf in column 7 (out finite there) and huge elsewhere
    gv, rv = bf16_val(got[5]), bf16_val(ref[5])
    same = (gv == rv) | (np.isnan(gv) & np.isnan(rv))
    assert same[7] and np.isinf(gv[7]), (gv[7], rv[7])
    assert np.array_equal(np.isfinite(gv), np.isfinite(rv))
    # the unfused GPU pair (GEMM into BF16 scratch, then bf16_scaled_add)
    d = g.gemm_bf16_nt(Ad, Bd)
    unfused = to_dev_bf16(out0)
    g.bf16_scaled_add(unfused, d, scale)
    check_bitexact16(got, bits16(unfused), f"fused vs unfused, non-finite {M}x{N}x{K}",
                     zero_sign=True)
