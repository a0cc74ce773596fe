"""Maximum sizes: outputs and workspaces past 2^31 elements / 2^32 bytes, so
that any 32-bit index or offset in a kernel, a launcher or a tensor map
would wrap.  Each case checks rows sampled on both sides of the crossing
(and the last row) against the oracle, and a guard band after the output."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import bf16_val, bits16, check_bitexact16, check_close16, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu
MAXDQ = 6.0 * 4.0
SENTINEL = 0x7BAD  # a finite bf16 / fp16 bit pattern no kernel output here takes


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_tcgen05_gb300 as lib
    yield lib
    assert lib.gemm_get_device_status() == 0


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def crossing_rows(total_rows, row_elems, seed):
    """Rows around the 2^31-element and 2^32-byte (16-bit) crossings, the
    first and last rows, and a few random ones."""
    cross = [(1 << 31) // row_elems]
    rows = {0, 1, total_rows - 1}
    for c in cross:
        rows.update(r for r in (c - 1, c, c + 1) if 0 <= r < total_rows)
    rng = np.random.default_rng(seed)
    rows.update(int(x) for x in rng.integers(0, total_rows, 4))
    return np.array(sorted(rows), dtype=np.int64)


def guarded(n_elems, dtype, guard=1 << 16):
    buf = torch.empty(n_elems + guard, dtype=dtype, device="cuda")
    buf[n_elems:].view(torch.int16).fill_(SENTINEL)
    return buf


def assert_guard_intact(buf, n_elems):
    tail = buf[n_elems:].view(torch.int16)
    assert bool(torch.all(tail == SENTINEL)), "write past the end of the output"


def amax(x):
    return float(np.abs(bf16_val(x)).max())


def test_bf16_nt_output_past_2_31_elements(g):
    M, N, K = 60000, 40960, 64
    A = synth.bf16_normal((M, K), 1.0, 701)
    B = synth.bf16_normal((N, K), 1.0, 702)
    buf = guarded(M * N, torch.bfloat16)
    C = buf[:M * N].view(M, N)
    g.gemm_bf16_nt(to_dev_bf16(A), to_dev_bf16(B), C)
    torch.cuda.synchronize()
    assert_guard_intact(buf, M * N)
    rows = crossing_rows(M, N, 703)
    got = bits16(C[torch.from_numpy(rows).cuda()])
    check_close16(got, oracle.gemm_bf16_nt(A, B, rows=rows), K, amax(A), amax(B),
                  what="bf16 past 2^31")


def test_scaled_acc_in_place_past_2_31_elements(g):
    M, N, K = 53248, 40960, 16
    A = synth.bf16_normal((M, K), 1.0, 711)
    B = synth.bf16_normal((N, K), 1.0, 712)
    base = to_dev_bf16(synth.scaled_acc_out(1, N, 713)).float()
    buf = guarded(M * N, torch.bfloat16)
    out = buf[:M * N].view(M, N)
    for r0 in range(0, M, 4096):  # old values differ from row to row
        r = torch.arange(r0, min(M, r0 + 4096), device="cuda")
        out[r0:r0 + len(r)] = (base + ((r % 7).float() * 0.25)[:, None]).bfloat16()
    rows = crossing_rows(M, N, 714)
    rows_d = torch.from_numpy(rows).cuda()
    old = bits16(out[rows_d])
    g.gemm_bf16_nt_scaled_acc(to_dev_bf16(A), to_dev_bf16(B), out, 0.37)
    torch.cuda.synchronize()
    assert_guard_intact(buf, M * N)
    ref = oracle.gemm_bf16_nt_scaled_acc(A, B, old, 0.37, rows=rows)
    check_close16(bits16(out[rows_d]), ref, K, amax(A), amax(B), what="scaled-acc past 2^31")


def test_nvfp4_output_past_2_31_elements(g):
    L, M, N, K = 1, 53248, 40960, 256
    a, b, sfa, sfb = synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, 721))
    buf = guarded(L * M * N, torch.float16)
    c = buf[:L * M * N]
    g.gemm_nvfp4_bs(to_dev_u8(a), to_dev_u8(b), to_dev_u8(sfa), to_dev_u8(sfb), L, M, N, K, c)
    torch.cuda.synchronize()
    assert_guard_intact(buf, L * M * N)
    rows = crossing_rows(L * M, N, 722)
    got = bits16(c.view(L * M, N)[torch.from_numpy(rows).cuda()])
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K, rows=rows)
    check_close16(got, ref, K, MAXDQ, MAXDQ, "f16", "nvfp4 past 2^31")


def test_bf16_splitk_workspace_past_4_gib(g):
    M, N, K, S = 16640, 16384, 1024, 4
    need = g.gemm_bf16_nt_splitk_workspace_bytes(M, N, K, S)
    assert need > (1 << 32)
    A = synth.bf16_normal((M, K), 1.0, 731)
    B = synth.bf16_normal((N, K), 1.0, 732)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    buf = guarded(M * N, torch.bfloat16)
    C = buf[:M * N].view(M, N)
    g.gemm_bf16_nt_splitk(to_dev_bf16(A), to_dev_bf16(B), S, workspace=ws, C=C)
    torch.cuda.synchronize()
    assert_guard_intact(buf, M * N)
    # partials [split][M][N] FP32: the last split's rows from 15616 on lie
    # past 2^32 bytes of the workspace
    rows = np.array([0, M // 2, 15615, 15616, 15617, M - 1], dtype=np.int64)
    got = bits16(C[torch.from_numpy(rows).cuda()])
    check_close16(got, oracle.gemm_bf16_nt(A, B, rows=rows), K, amax(A), amax(B),
                  what="split-K workspace past 4 GiB")


def test_nvfp4_splitk_workspace_past_4_gib(g):
    L, M, N, K, S = 2, 1024, 132096, 1024, 4
    need = L * g.gemm_nvfp4_bs_splitk_workspace_bytes(M, N, K, S)
    assert need > (1 << 32)
    a, b, sfa, sfb = synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, 741))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    buf = guarded(L * M * N, torch.float16)
    c = buf[:L * M * N]
    g.gemm_nvfp4_bs_splitk(to_dev_u8(a), to_dev_u8(b), to_dev_u8(sfa), to_dev_u8(sfb), M, N, K, S,
                           workspace=ws, c=c, L=L)
    torch.cuda.synchronize()
    assert_guard_intact(buf, L * M * N)
    rows = np.array([0, 511, M - 1, M, M + 700, 2 * M - 1], dtype=np.int64)
    got = bits16(c.view(L * M, N)[torch.from_numpy(rows).cuda()])
    ref = oracle.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K, rows=rows)
    check_close16(got, ref, K, MAXDQ, MAXDQ, "f16", "nvfp4 split-K workspace past 4 GiB")


def test_w4a16_weights_past_2_31_elements(g):
    # N x K > 2^31 weights: 1 GiB of codes, a 4.3 GB converted workspace
    M, N, K = 3, 131328, 16384
    A, b, sfb, scale2 = synth.w4a16_inputs(synth.W4a16("t", M, N, K, 0.05, 751))
    Ad, bd, sd = to_dev_bf16(A), to_dev_u8(b), to_dev_u8(sfb)
    fused = bits16(g.gemm_w4a16(Ad, bd, sd, scale2))
    ws = torch.empty(g.gemm_w4a16_ws_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    assert ws.numel() > (1 << 32)
    two = bits16(g.gemm_w4a16_ws(Ad, bd, sd, scale2, ws))
    assert np.array_equal(fused, two), "two-pass differs from fused past 2^31 weights"
    # the last weight rows sit past 2^31 elements of the workspace: read them
    # back through one-hot activations (row m picks weight k = m)
    W_last = ws.view(torch.int16).view(N, K)[N - 2:].cpu().numpy().view(np.uint16)
    eye = np.zeros((K, K), dtype=np.uint16)
    eye[np.arange(K), np.arange(K)] = 0x3F80
    # (a one-hot sum turns a -0 weight into +0: signed zeros compare equal)
    ref_w = oracle.gemm_w4a16(eye, b[N - 2:], sfb[N - 2:], 1.0)  # [K][2]
    check_bitexact16(W_last.T.copy(), ref_w, "converted weights past 2^31")
    rows = np.array([0, M - 1], dtype=np.int64)
    tab = np.abs(np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0] * 2))
    sc = torch.from_numpy(sfb.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    wmax = float(tab.max() * sc.max() * abs(scale2))
    check_close16(fused[rows], oracle.gemm_w4a16(A, b, sfb, scale2, rows=rows), K, amax(A), wmax,
                  what="w4a16 past 2^31 weights")
