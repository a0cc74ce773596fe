"""The failure path on the GPU, without a fault: a bounded wait that runs
out sets the device status word, the status call reports and clears it,
and the context keeps working."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from nvfp4_block_scaled_tcgen05_gb300 import synth
from parity import bf16_val, bits16, check_close16, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_block_scaled_tcgen05_gb300 as lib
    return lib


def test_wait_timeout_is_reported_and_cleared(g):
    assert g.gemm_get_device_status() == 0
    g.gemm_selftest_wait_timeout(50)
    assert g.gemm_get_device_status() == 7   # GEMM_ERR_TIMEOUT
    assert g.gemm_get_device_status() == 0   # cleared by the read
    # the context still runs GEMMs correctly
    A = synth.bf16_normal((256, 64), 1.0, 5)
    B = synth.bf16_normal((512, 64), 1.0, 6)
    C = g.gemm_bf16_nt(to_dev_bf16(A), to_dev_bf16(B))
    amax = float(np.abs(bf16_val(A)).max()) * float(np.abs(bf16_val(B)).max())
    check_close16(bits16(C), oracle.gemm_bf16_nt(A, B), 64, amax, 1.0, what="after timeout")
    assert g.gemm_get_device_status() == 0


def test_selftest_rejects_bad_limit(g):
    with pytest.raises(g.GemmError):
        g.gemm_selftest_wait_timeout(0)


_CAPTURE_CHILD = r"""
import torch
import nvfp4_block_scaled_tcgen05_gb300 as g
lib = g.load()
A = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
B = torch.zeros((256, 64), dtype=torch.bfloat16, device="cuda")
C = torch.empty((128, 256), dtype=torch.bfloat16, device="cuda")
s = torch.cuda.Stream()
torch.cuda.synchronize()
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph, stream=s):
    rc_capture = lib.gemm_bf16_nt(A.data_ptr(), B.data_ptr(), C.data_ptr(), 128, 256, 64,
                                  s.cuda_stream)
rc_after = lib.gemm_bf16_nt(A.data_ptr(), B.data_ptr(), C.data_ptr(), 128, 256, 64, None)
torch.cuda.synchronize()
print("RC", rc_capture, rc_after, int(C.float().abs().sum().item()))
"""


def test_first_call_during_capture_is_refused(g):
    # A fresh process whose first library call comes inside a stream capture:
    # the one-time device set-up may not run there, so the call returns
    # GEMM_ERR_CAPTURE (9) without enqueuing anything; the next call outside
    # the capture does the set-up and runs.
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CAPTURE_CHILD], cwd=root, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("RC ")][-1]
    assert line.split()[1:] == ["9", "0", "0"], line
