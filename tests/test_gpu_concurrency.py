"""Host threads calling the library at the same time, each on a stream of
its own: the one-time device set-up happens once whoever comes first, and
every call's result equals the same call made alone (the kernels of the two
streams share the GPU but no state)."""
from __future__ import annotations

import os
import subprocess
import sys
import threading

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


def _bits(t):
    return t.detach().contiguous().view(torch.uint8).cpu().numpy().copy()


def test_two_threads_two_streams_match_calls_made_alone(g):
    A = to_dev_bf16(synth.bf16_normal((520, 1024), 1.0, 1))
    B = to_dev_bf16(synth.bf16_normal((776, 1024), 1.0, 2))
    L, M, N, K, S = 2, 128, 512, 2048, 4
    fa, fb, fsa, fsb = [to_dev_u8(x) for x in synth.nvfp4_inputs(synth.Nvfp4("t", L, M, N, K, 3))]
    wa, wb, wsfb, s2 = synth.w4a16_inputs(synth.W4a16("t", 300, 520, 768, 0.5, 4))
    wa, wb, wsfb = to_dev_bf16(wa), to_dev_u8(wb), to_dev_u8(wsfb)

    ref_bf16 = _bits(g.gemm_bf16_nt(A, B))
    ref_fp4 = _bits(g.gemm_nvfp4_bs_splitk(fa, fb, fsa, fsb, M, N, K, S, L=L))
    ref_w4 = _bits(g.gemm_w4a16(wa, wb, wsfb, s2))
    torch.cuda.synchronize()

    results, errors = {}, []

    def worker_a():
        try:
            s = torch.cuda.Stream()
            C = torch.empty((520, 776), dtype=torch.bfloat16, device="cuda")
            for _ in range(40):
                g.gemm_bf16_nt(A, B, C, stream=s)
            s.synchronize()
            results["bf16"] = _bits(C)
        except Exception as e:  # reported by the main thread
            errors.append(e)

    def worker_b():
        try:
            s = torch.cuda.Stream()
            ws = torch.empty(L * g.gemm_nvfp4_bs_splitk_workspace_bytes(M, N, K, S),
                             dtype=torch.uint8, device="cuda")
            c = torch.empty((L, M, N), dtype=torch.float16, device="cuda")
            C2 = torch.empty((300, 520), dtype=torch.bfloat16, device="cuda")
            for _ in range(40):
                g.gemm_nvfp4_bs_splitk(fa, fb, fsa, fsb, M, N, K, S, workspace=ws, c=c, stream=s,
                                       L=L)
                g.gemm_w4a16(wa, wb, wsfb, s2, C2, stream=s)
            s.synchronize()
            results["fp4"] = _bits(c)
            results["w4"] = _bits(C2)
        except Exception as e:
            errors.append(e)

    threads = [threading.Thread(target=worker_a), threading.Thread(target=worker_b)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    assert np.array_equal(results["bf16"], ref_bf16)
    assert np.array_equal(results["fp4"], ref_fp4)
    assert np.array_equal(results["w4"], ref_w4)
    assert g.gemm_get_device_status() == 0


_FIRST_CALLS_CHILD = r"""
import threading, torch
import nvfp4_block_scaled_tcgen05_gb300 as g
torch.cuda.init()
A = torch.ones((256, 256), dtype=torch.bfloat16, device="cuda")
torch.cuda.synchronize()
go = threading.Barrier(4)
out, errs = [None] * 4, []
def first_call(i):
    try:
        s = torch.cuda.Stream()
        go.wait()
        C = g.gemm_bf16_nt(A, A, stream=s)   # every thread's first library call
        s.synchronize()
        out[i] = float(C.float().sum().item())
    except Exception as e:
        errs.append(repr(e))
ts = [threading.Thread(target=first_call, args=(i,)) for i in range(4)]
[t.start() for t in ts]
[t.join() for t in ts]
print("ERRS", errs)
print("SUMS", out, g.gemm_get_device_status())
"""


def test_first_calls_from_four_threads_at_once(g):
    # a fresh process whose first four library calls race each other: the
    # device set-up runs once and every call succeeds
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALLS_CHILD], cwd=root, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = {ln.split()[0]: ln for ln in r.stdout.splitlines() if ln.split()}
    assert lines["ERRS"] == "ERRS []", lines["ERRS"]
    # ones(256 x 256) . ones^T = 256 everywhere: sum 256^3
    assert lines["SUMS"] == f"SUMS {[float(256 ** 3)] * 4} 0", lines["SUMS"]
