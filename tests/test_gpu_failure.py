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
