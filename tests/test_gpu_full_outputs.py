"""Every output element of the full-size problems against the oracle (the
other full-size tests sample rows): the BF16 GEMMs at gate/up, down, qkv and
gqa through the default entry point, gate/up in the NN layout, down and qkv
through stream-K, gqa through split-K, the NVFP4 decode shapes through
split-K, and W4A16 at qkvz (~45 s of oracle on 16 host cores).  The NVFP4
GEMM at 4096 x 7168 x 16384 takes the oracle ~5 minutes and runs only with
--slow-oracle (its rows are sampled in the NVFP4 tests)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import bf16_val, bits16, check_close16, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu
MAXDQ = 6.0 * 4.0
E2M1_ABS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0] * 2)


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_tcgen05_gb300 as lib
    yield lib
    assert lib.gemm_get_device_status() == 0


def amax(x):
    return float(np.abs(bf16_val(x)).max())


def check_all(got, ref, K, a_max, b_max, fmt, what, rows_per_chunk=512):
    """The 1-ULP-or-absolute rule on every element, a block of rows at a time."""
    assert got.shape == ref.shape
    exact = 0
    worst = 0
    for r0 in range(0, got.shape[0], rows_per_chunk):
        st = check_close16(got[r0:r0 + rows_per_chunk], ref[r0:r0 + rows_per_chunk], K, a_max,
                           b_max, fmt, f"{what} rows {r0}..")
        exact += st["frac_exact"] * got[r0:r0 + rows_per_chunk].size
        worst = max(worst, st["max_ulp"])
    return {"frac_exact": exact / got.size, "max_ulp": worst}


@pytest.mark.parametrize("name", ["gateup", "down", "qkv", "gqa"])
def test_bf16_every_output(g, name):
    w = synth.BF16_WORKLOADS[name]
    A, B = synth.gemm_inputs(w)
    got = bits16(g.gemm_bf16_nt(to_dev_bf16(A), to_dev_bf16(B)))
    ref = oracle.gemm_bf16_nt(A, B)
    stats = check_all(got, ref, w.K, amax(A), amax(B), "bf16", name)
    assert stats["frac_exact"] > 0.9, stats


def test_bf16_nn_gateup_every_output(g):
    # B stored [K][N]: the oracle takes it back to [N][K]
    w = synth.BF16_WORKLOADS["gateup"]
    A, B = synth.gemm_inputs(w)
    Bt = np.ascontiguousarray(B.T)
    got = bits16(g.gemm_bf16_nn(to_dev_bf16(A), to_dev_bf16(Bt)))
    stats = check_all(got, oracle.gemm_bf16_nt(A, B), w.K, amax(A), amax(B), "bf16", "nn gateup")
    assert stats["frac_exact"] > 0.9, stats


@pytest.mark.parametrize("name", ["down", "qkv"])
def test_bf16_streamk_every_output(g, name):
    w = synth.BF16_WORKLOADS[name]
    A, B = synth.gemm_inputs(w)
    got = bits16(g.gemm_bf16_nt_streamk(to_dev_bf16(A), to_dev_bf16(B)))
    stats = check_all(got, oracle.gemm_bf16_nt(A, B), w.K, amax(A), amax(B), "bf16",
                      f"{name} stream-K")
    assert stats["frac_exact"] > 0.9, stats


def test_bf16_splitk_gqa_every_output(g):
    w = synth.BF16_WORKLOADS["gqa"]
    A, B = synth.gemm_inputs(w)
    got = bits16(g.gemm_bf16_nt_splitk(to_dev_bf16(A), to_dev_bf16(B), 4))
    stats = check_all(got, oracle.gemm_bf16_nt(A, B), w.K, amax(A), amax(B), "bf16",
                      "gqa split-K 4")
    assert stats["frac_exact"] > 0.9, stats


@pytest.mark.slow_oracle  # ~5 minutes of oracle on 16 host cores
def test_nvfp4_every_output(g):
    w = synth.NVFP4
    a, b, sfa, sfb = synth.nvfp4_inputs(w)
    c = g.gemm_nvfp4_bs(to_dev_u8(a), to_dev_u8(b), to_dev_u8(sfa), to_dev_u8(sfb), w.L, w.M, w.N,
                        w.K)
    got = bits16(c).reshape(w.L * w.M, w.N)
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, w.L, w.M, w.N, w.K)
    stats = check_all(got, ref, w.K, MAXDQ, MAXDQ, "f16", "nvfp4 4096x7168x16384")
    assert stats["frac_exact"] > 0.9, stats


@pytest.mark.parametrize("name", sorted(synth.NVFP4_DECODE))
def test_nvfp4_decode_every_output(g, name):
    w, splits = synth.NVFP4_DECODE[name]
    a, b, sfa, sfb = synth.nvfp4_inputs(w)
    c = g.gemm_nvfp4_bs_splitk(to_dev_u8(a), to_dev_u8(b), to_dev_u8(sfa), to_dev_u8(sfb), w.M,
                               w.N, w.K, splits)
    got = bits16(c).reshape(w.M, w.N)
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, w.L, w.M, w.N, w.K)
    stats = check_all(got, ref, w.K, MAXDQ, MAXDQ, "f16", name)
    assert stats["frac_exact"] > 0.9, stats


def test_w4a16_qkvz_every_output(g):
    w = synth.W4A16["w4a16_qkvz"]
    A, b, sfb, scale2 = synth.w4a16_inputs(w)
    got = bits16(g.gemm_w4a16(to_dev_bf16(A), to_dev_u8(b), to_dev_u8(sfb), scale2))
    ref = oracle.gemm_w4a16(A, b, sfb, scale2)
    sc = torch.from_numpy(sfb.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    wmax = float(E2M1_ABS.max() * sc.max() * abs(scale2))
    stats = check_all(got, ref, w.K, amax(A), wmax, "bf16", "w4a16 qkvz")
    assert stats["frac_exact"] > 0.9, stats
