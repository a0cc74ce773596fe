"""Every entry point captured into a CUDA graph: the captured call enqueues
only device work (no allocation, copy, host synchronisation or set-up), a
replay writes the same bits as the eager call, and a replay after the
inputs' contents changed in place equals an eager call on the new
contents (nothing of the data is baked in at capture time)."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import to_dev_bf16, to_dev_u8

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


def _bf16(shape, seed, sigma=1.0):
    return to_dev_bf16(synth.bf16_normal(shape, sigma, seed))


def _refill_bf16(t, seed):
    t.copy_(_bf16(tuple(t.shape), seed))


def _refill_u8(t, seed):
    t.copy_(to_dev_u8(synth.uniform_bytes(t.numel(), seed).reshape(tuple(t.shape))))


def case_bf16_nt(g):
    A, B = _bf16((520, 1024), 1), _bf16((776, 1024), 2)
    C = torch.empty((520, 776), dtype=torch.bfloat16, device="cuda")
    return dict(run=lambda s: g.gemm_bf16_nt(A, B, C, stream=s), outs=[C],
                mutate=lambda k: _refill_bf16(A, 10 + k))


def case_bf16_nn(g):
    A, B = _bf16((520, 1024), 3), _bf16((1024, 776), 4)
    C = torch.empty((520, 776), dtype=torch.bfloat16, device="cuda")
    return dict(run=lambda s: g.gemm_bf16_nn(A, B, C, stream=s), outs=[C],
                mutate=lambda k: _refill_bf16(B, 20 + k))


def case_scaled_acc(g):
    # in place: the replay starts from the same old output each time
    A, B = _bf16((512, 16), 5), _bf16((1032, 16), 6)
    init = to_dev_bf16(synth.scaled_acc_out(512, 1032, 7))
    C = init.clone()
    return dict(run=lambda s: g.gemm_bf16_nt_scaled_acc(A, B, C, 0.37, stream=s), outs=[C],
                reset=lambda: C.copy_(init), mutate=lambda k: _refill_bf16(A, 30 + k))


def case_ordered(g):
    A, B = _bf16((300, 512), 8), _bf16((256, 512), 9)
    C = torch.empty((300, 256), dtype=torch.float32, device="cuda")
    return dict(run=lambda s: g.gemm_bf16_nt_ordered(A, B, C, stream=s), outs=[C],
                mutate=lambda k: _refill_bf16(A, 40 + k))


def case_splitk(g):
    M, N, K, S = 384, 512, 2048, 3
    A, B = _bf16((M, K), 11), _bf16((N, K), 12)
    ws = torch.empty(g.gemm_bf16_nt_splitk_workspace_bytes(M, N, K, S), dtype=torch.uint8,
                     device="cuda")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    return dict(run=lambda s: g.gemm_bf16_nt_splitk(A, B, S, workspace=ws, C=C, stream=s),
                outs=[C], mutate=lambda k: _refill_bf16(B, 50 + k))


def case_splitk_static(g):
    from nvfp4_block_scaled_tcgen05_gb300 import binding
    so = ctypes.CDLL(binding.library_path())
    f = so.gemm_bf16_nt_splitk_static
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    M, N, K, S = 384, 512, 2048, 4
    A, B = _bf16((M, K), 13), _bf16((N, K), 14)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def run(s):
        assert f(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, S, s.cuda_stream) == 0
    return dict(run=run, outs=[C], mutate=lambda k: _refill_bf16(A, 60 + k))


def case_streamk(g):
    M, N, K = 600, 1032, 2048
    A, B = _bf16((M, K), 15), _bf16((N, K), 16)
    ws = torch.empty(max(g.gemm_bf16_nt_streamk_workspace_bytes(), 16), dtype=torch.uint8,
                     device="cuda")
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    return dict(run=lambda s: g.gemm_bf16_nt_streamk(A, B, workspace=ws, C=C, stream=s),
                outs=[C], mutate=lambda k: _refill_bf16(A, 70 + k))


def _w4(M, N, K, seed):
    A, b, sfb, scale2 = synth.w4a16_inputs(synth.W4a16("t", M, N, K, 0.25, seed))
    return to_dev_bf16(A), to_dev_u8(b), to_dev_u8(sfb), scale2


def case_w4a16(g):
    A, b, sfb, scale2 = _w4(520, 776, 512, 17)
    C = torch.empty((520, 776), dtype=torch.bfloat16, device="cuda")
    return dict(run=lambda s: g.gemm_w4a16(A, b, sfb, scale2, C, stream=s), outs=[C],
                mutate=lambda k: _refill_u8(b, 80 + k))


def case_w4a16_t(g):
    M, N, K, ldb = 300, 264, 512, 384
    A, b, sfb, scale2 = _w4(M, N, K, 18)
    b_t = torch.zeros((K // 2, ldb), dtype=torch.uint8, device="cuda")
    sfb_t = torch.full((K // 16, ldb), 0x38, dtype=torch.uint8, device="cuda")
    b_t[:, :N] = b.t()
    sfb_t[:, :N] = sfb.t()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    return dict(run=lambda s: g.gemm_w4a16_t(A, b_t, sfb_t, scale2, N, C, stream=s), outs=[C],
                mutate=lambda k: _refill_bf16(A, 90 + k))


def case_w4a16_ws(g):
    A, b, sfb, scale2 = _w4(520, 776, 512, 19)
    ws = torch.empty(g.gemm_w4a16_ws_workspace_bytes(776, 512), dtype=torch.uint8, device="cuda")
    C = torch.empty((520, 776), dtype=torch.bfloat16, device="cuda")
    return dict(run=lambda s: g.gemm_w4a16_ws(A, b, sfb, scale2, workspace=ws, C=C, stream=s),
                outs=[C, ws], mutate=lambda k: _refill_u8(b, 100 + k))


def _fp4(L, M, N, K, seed):
    return [to_dev_u8(x) for x in synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, seed))]


def case_nvfp4(g):
    L, M, N, K = 2, 256, 512, 1024
    a, b, sfa, sfb = _fp4(L, M, N, K, 21)
    c = torch.empty((L, M, N), dtype=torch.float16, device="cuda")
    return dict(run=lambda s: g.gemm_nvfp4_bs(a, b, sfa, sfb, L, M, N, K, c, stream=s), outs=[c],
                mutate=lambda k: _refill_u8(a, 110 + k))


def case_nvfp4_splitk_batched(g):
    L, M, N, K, S = 2, 128, 512, 2048, 4
    a, b, sfa, sfb = _fp4(L, M, N, K, 22)
    ws = torch.empty(L * g.gemm_nvfp4_bs_splitk_workspace_bytes(M, N, K, S), dtype=torch.uint8,
                     device="cuda")
    c = torch.empty((L, M, N), dtype=torch.float16, device="cuda")
    return dict(run=lambda s: g.gemm_nvfp4_bs_splitk(a, b, sfa, sfb, M, N, K, S, workspace=ws,
                                                      c=c, stream=s, L=L),
                outs=[c], mutate=lambda k: _refill_u8(b, 120 + k))


def case_scaled_add(g):
    init = to_dev_bf16(synth.scaled_acc_out(300, 1000, 23))
    out = init.clone()
    d = _bf16((300, 1000), 24)
    return dict(run=lambda s: g.bf16_scaled_add(out, d, -0.75, stream=s), outs=[out],
                reset=lambda: out.copy_(init), mutate=lambda k: _refill_bf16(d, 130 + k))


CASES = {f.__name__[5:]: f for f in (
    case_bf16_nt, case_bf16_nn, case_scaled_acc, case_ordered, case_splitk, case_splitk_static,
    case_streamk, case_w4a16, case_w4a16_t, case_w4a16_ws, case_nvfp4, case_nvfp4_splitk_batched,
    case_scaled_add)}


def _bits(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy().copy()


@pytest.mark.parametrize("name", sorted(CASES))
def test_graph_replay_equals_eager(g, name):
    c = CASES[name](g)
    run, outs = c["run"], c["outs"]
    reset = c.get("reset", lambda: None)
    in_place = "reset" in c
    s = torch.cuda.Stream()

    def scrub():
        # outputs that are not also inputs hold junk before each replay, so
        # a replay that wrote nothing cannot pass
        if in_place:
            reset()
        else:
            for o in outs:
                o.view(torch.uint8).fill_(0xA5)

    torch.cuda.synchronize()
    reset()
    run(s)
    s.synchronize()
    eager = [_bits(o) for o in outs]

    graph = torch.cuda.CUDAGraph()
    reset()
    with torch.cuda.graph(graph, stream=s):
        run(s)
    torch.cuda.synchronize()
    for rep in range(2):
        scrub()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        for o, ref in zip(outs, eager):
            assert np.array_equal(_bits(o), ref), f"{name}: replay {rep} differs from eager"

    # new input contents, same buffers: the replay follows the data
    for k in range(2):
        c["mutate"](k)
        scrub()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        got = [_bits(o) for o in outs]
        reset()
        run(s)
        s.synchronize()
        for o, gb in zip(outs, got):
            assert np.array_equal(_bits(o), gb), f"{name}: replay on new inputs {k} differs"
        assert not all(np.array_equal(gb, e) for gb, e in zip(got, eager)), \
            f"{name}: new inputs left every output unchanged"
    assert g.gemm_get_device_status() == 0
