"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/gb300gemm.h declares, and rejects bad
arguments before touching the device."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gb300gemm.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_block_scaled_tcgen05_gb300 import build, binding
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"GB300GEMM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"gemm_bf16_nt", "gemm_bf16_nt_scaled_acc", "gemm_bf16_nt_ordered", "gemm_nvfp4_bs",
            "bf16_scaled_add", "gemm_get_device_status", "gemm_status_string"} <= names


def test_library_exports_every_declared_symbol(lib):
    from nvfp4_block_scaled_tcgen05_gb300 import binding
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "gb300gemm.h"\nint main(void){return gemm_status_string(0)[0]==0;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I",
                    os.path.join(ROOT, "include"), str(src)], check=True)


def test_status_strings(lib):
    for code in range(9):
        s = lib.gemm_status_string(code).decode()
        assert s.startswith("GEMM_")
    assert lib.gemm_status_string(99).decode() == "unknown status"


P = 0x10000  # a 16-byte aligned fake address; validation never dereferences it


@pytest.mark.parametrize("args,expect", [
    ((0, P, 2 * P, 8, 8, 8), 1),                 # NULL A
    ((P, 0, 2 * P, 8, 8, 8), 1),                 # NULL B
    ((P, 2 * P, 0, 8, 8, 8), 1),                 # NULL C
    ((P, 2 * P, 3 * P, 0, 8, 8), 2),             # M = 0
    ((P, 2 * P, 3 * P, 8, -1, 8), 2),            # N < 0
    ((P, 2 * P, 3 * P, 8, 8, 0), 2),             # K = 0
    ((P + 8, 2 * P, 3 * P, 8, 8, 8), 3),         # misaligned A
    ((P, 2 * P, 3 * P, 8, 8, 12), 3),            # K % 8 != 0
    ((P, 2 * P, 3 * P, 8, 12, 8), 3),            # N % 8 != 0 (C pitch)
    ((P, 2 * P, P + 64, 8, 8, 8), 4),            # C overlaps A
])
def test_gemm_bf16_nt_rejects_bad_arguments(lib, args, expect):
    assert lib.gemm_bf16_nt(*args, None) == expect
    assert lib.gemm_bf16_nt_scaled_acc(*args, ctypes.c_float(1.0), None) == expect


def test_router_rejects_bad_arguments(lib):
    assert lib.gemm_bf16_nt_ordered(0, P, 2 * P, 8, 8, 8, None) == 1
    assert lib.gemm_bf16_nt_ordered(P, 2 * P, 3 * P, 8, 8, 0, None) == 2
    assert lib.gemm_bf16_nt_ordered(P, 2 * P, 3 * P, 8, 8, 4, None) == 3
    assert lib.gemm_bf16_nt_ordered(P, 2 * P, 2 * P + 16, 8, 8, 8, None) == 4


@pytest.mark.parametrize("dims,expect", [
    ((0, 128, 128, 256), 2),
    ((1, 100, 128, 256), 2),      # M % 128
    ((1, 128, 200, 256), 2),      # N % 128
    ((1, 128, 128, 128), 2),      # K % 256
])
def test_nvfp4_shape_rules(lib, dims, expect):
    assert lib.gemm_nvfp4_bs(P, 2 * P, 3 * P, 4 * P, 5 * P, *dims, None) == expect


# Valid arguments with fake pointers get past validation: only where no GPU
# is present can such a call run (it then stops at the device query); on a
# GPU it would launch a kernel on the fake addresses.
@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="a GPU is present")
def test_valid_nvfp4_call_without_a_gpu_reports_no_device(lib):
    assert lib.gemm_nvfp4_bs(P, 2 * P, 3 * P, 4 * P, 5 * P, 1, 128, 128, 256, None) == 8


def test_nvfp4_pointer_rules(lib):
    assert lib.gemm_nvfp4_bs(P, 2 * P, 0, 4 * P, 5 * P, 1, 128, 128, 256, None) == 1
    assert lib.gemm_nvfp4_bs(P, 2 * P, 3 * P + 4, 4 * P, 5 * P, 1, 128, 128, 256, None) == 3
    # c overlapping sfb
    assert lib.gemm_nvfp4_bs(P, 2 * P, 3 * P, 4 * P, 4 * P + 1024, 1, 128, 128, 256, None) == 4


def test_scaled_add_rules(lib):
    f = ctypes.c_float(1.0)
    assert lib.bf16_scaled_add(0, P, f, 10, None) == 1
    assert lib.bf16_scaled_add(P, 2 * P, f, 0, None) == 2
    assert lib.bf16_scaled_add(P + 2, 2 * P, f, 10, None) == 3
    assert lib.bf16_scaled_add(P, P + 16, f, 10, None) == 4


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="a GPU is present")
def test_valid_call_without_a_gpu_reports_no_device(lib):
    assert lib.gemm_bf16_nt(P, 2 * P, 3 * P, 8, 8, 8, None) == 8


def test_splitk_workspace_size_rules(lib):
    ws = lib.gemm_bf16_nt_splitk_workspace_bytes
    ws.restype = ctypes.c_size_t
    assert ws(5120, 512, 2048, 4) == 4 * 5120 * 512 * 4
    assert ws(300, 520, 200, 3) == 2 * 300 * 520 * 4   # 4 K blocks: 2 per split, 2 splits
    assert ws(64, 64, 64, 8) == 1 * 64 * 64 * 4        # one K block: one split
    assert ws(0, 8, 8, 1) == 0 and ws(8, 8, 8, 0) == 0 and ws(8, 8, 8, 65) == 0


def test_splitk_rejects_bad_arguments(lib):
    f = lib.gemm_bf16_nt_splitk
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_size_t] + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    big = 1 << 30
    assert f(P, 2 * P, 3 * P, 0, big, 8, 8, 64, 2, None) == 1          # NULL workspace
    assert f(P, 2 * P, 3 * P, 4 * P, big, 8, 8, 64, 0, None) == 2      # k_splits < 1
    assert f(P, 2 * P, 3 * P, 4 * P, 16, 64, 64, 256, 2, None) == 2    # workspace too small
    assert f(P, 2 * P, 3 * P, 4 * P + 8, big, 8, 8, 64, 2, None) == 3  # misaligned workspace
    assert f(P, 2 * P, 3 * P, P + 16, big, 8, 8, 64, 2, None) == 4     # workspace overlaps A


def test_nvfp4_splitk_workspace_size_rules(lib):
    ws = lib.gemm_nvfp4_bs_splitk_workspace_bytes
    ws.restype = ctypes.c_size_t
    assert ws(128, 7168, 16384, 5) == 5 * 128 * 7168 * 4      # 64 blocks: 13 per split, 5 splits
    assert ws(128, 4096, 7168, 7) == 7 * 128 * 4096 * 4       # 28 blocks: 4 per split
    assert ws(128, 256, 1024, 3) == 2 * 128 * 256 * 4         # 4 blocks: 2 per split, 2 splits
    assert ws(128, 256, 512, 64) == 2 * 128 * 256 * 4         # capped at K/256 = 2
    assert ws(128, 256, 1000, 2) == 0 and ws(128, 256, 1024, 0) == 0 and ws(0, 256, 1024, 2) == 0


def test_nvfp4_splitk_rejects_bad_arguments(lib):
    f = lib.gemm_nvfp4_bs_splitk
    f.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_size_t] + [ctypes.c_int] * 5 + [ctypes.c_void_p]
    big = 1 << 30
    ok = (P, 2 * P, 3 * P, 4 * P, 5 * P, 6 * P, big)
    assert f(P, 2 * P, 3 * P, 4 * P, 5 * P, 0, big, 1, 128, 256, 1024, 2, None) == 1  # NULL ws
    assert f(*ok, 0, 128, 256, 1024, 2, None) == 2            # L = 0
    # L = 2 needs twice the per-batch workspace
    per_batch = 2 * 128 * 256 * 4
    assert f(P, 2 * P, 3 * P, 4 * P, 5 * P, 6 * P, 2 * per_batch - 16, 2, 128, 256, 1024, 2,
             None) == 2
    assert f(*ok, 1, 100, 256, 1024, 2, None) == 2            # M % 128
    assert f(*ok, 1, 128, 256, 1000, 2, None) == 2            # K % 256
    assert f(*ok, 1, 128, 256, 1024, 0, None) == 2            # k_splits < 1
    assert f(*ok, 1, 128, 256, 1024, 65, None) == 2           # k_splits > 64
    assert f(P, 2 * P, 3 * P, 4 * P, 5 * P, 6 * P, 16, 1, 128, 256, 1024, 2, None) == 2  # small ws
    assert f(P, 2 * P, 3 * P, 4 * P, 5 * P, 6 * P + 8, big, 1, 128, 256, 1024, 2, None) == 3
    assert f(P, 2 * P, 3 * P, 4 * P, 5 * P, P + 16, big, 1, 128, 256, 1024, 2, None) == 4  # ws on a


@pytest.mark.parametrize("args,expect", [
    ((0, P, 2 * P, 8, 8, 8), 1),                 # NULL A
    ((P, 2 * P, 3 * P, 0, 8, 8), 2),             # M = 0
    ((P + 8, 2 * P, 3 * P, 8, 8, 8), 3),         # misaligned A
    ((P, 2 * P, 3 * P, 8, 8, 12), 3),            # K % 8 != 0 (A pitch)
    ((P, 2 * P, 3 * P, 8, 12, 8), 3),            # N % 8 != 0 (B and C pitch)
    ((P, 2 * P, 2 * P + 16, 8, 8, 8), 4),        # C overlaps B
])
def test_gemm_bf16_nn_rejects_bad_arguments(lib, args, expect):
    assert lib.gemm_bf16_nn(*args, None) == expect


def test_streamk_rejects_bad_arguments(lib):
    f = lib.gemm_bf16_nt_streamk
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_size_t] + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    big = 1 << 20
    assert f(0, 2 * P, 3 * P, 4 * P, big, 8, 8, 64, None) == 1            # NULL A
    assert f(P, 2 * P, 3 * P, 0, big, 8, 8, 64, None) == 1                # NULL workspace
    assert f(P, 2 * P, 3 * P, 4 * P, big, 0, 8, 64, None) == 2            # M = 0
    assert f(P, 2 * P, 3 * P, 4 * P + 8, big, 8, 8, 64, None) == 3        # misaligned workspace
    assert f(P, 2 * P, 3 * P, 4 * P, big, 8, 12, 64, None) == 3           # N % 8
    assert f(P, 2 * P, 3 * P, P + 16, big, 8, 8, 64, None) == 4           # workspace overlaps A
    assert f(P, 2 * P, 3 * P, 3 * P - 16, big, 8, 8, 64, None) == 4       # ... or C


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="a GPU is present")
def test_streamk_workspace_without_a_gpu(lib):
    ws = lib.gemm_bf16_nt_streamk_workspace_bytes
    ws.restype = ctypes.c_size_t
    assert ws() == 0
    f = lib.gemm_bf16_nt_streamk
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_size_t] + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    assert f(P, 2 * P, 3 * P, 8 * P, 1 << 20, 8, 8, 64, None) == 8


@pytest.mark.parametrize("args,expect", [
    ((0, 2 * P, 3 * P, 1.0, 4 * P, 8, 8, 256), 1),         # NULL A
    ((P, 2 * P, 0, 1.0, 4 * P, 8, 8, 256), 1),             # NULL scales
    ((P, 2 * P, 3 * P, 1.0, 4 * P, 0, 8, 256), 2),         # M = 0
    ((P, 2 * P + 8, 3 * P, 1.0, 4 * P, 8, 8, 256), 3),     # misaligned b
    ((P, 2 * P, 3 * P, 1.0, 4 * P, 8, 8, 224), 3),         # K % 256 != 0
    ((P, 2 * P, 3 * P, 1.0, 4 * P, 8, 12, 256), 3),        # N % 8 != 0
    ((P, 2 * P, 3 * P, 1.0, 2 * P + 16, 8, 8, 256), 4),    # C overlaps b
    ((P, 2 * P, 3 * P, 1.0, P + 16, 8, 8, 256), 4),        # C overlaps A
])
def test_w4a16_rejects_bad_arguments(lib, args, expect):
    f = lib.gemm_w4a16
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_float, ctypes.c_void_p] + [ctypes.c_int] * 3 + \
        [ctypes.c_void_p]
    assert f(*args, None) == expect


def test_w4a16_ws_workspace_and_arguments(lib):
    ws = lib.gemm_w4a16_ws_workspace_bytes
    ws.restype = ctypes.c_size_t
    assert ws(12288, 2048) == 12288 * 2048 * 2
    assert ws(8, 224) == 0 and ws(0, 256) == 0
    f = lib.gemm_w4a16_ws
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_float] + [ctypes.c_void_p] * 2 + \
        [ctypes.c_size_t] + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    big = 1 << 20
    assert f(P, 2 * P, 3 * P, 1.0, 4 * P, 0, big, 8, 8, 256, None) == 1           # NULL workspace
    assert f(P, 2 * P, 3 * P, 1.0, 4 * P, 5 * P + 8, big, 8, 8, 256, None) == 3   # misaligned
    assert f(P, 2 * P, 3 * P, 1.0, 4 * P, 5 * P, 16, 8, 8, 256, None) == 2        # too small
    assert f(P, 2 * P, 3 * P, 1.0, 4 * P, 4 * P + 16, big, 8, 8, 256, None) == 4  # on C


@pytest.mark.parametrize("args,expect", [
    ((0, 2 * P, 3 * P, 1.0, 4 * P, 8, 8, 128, 16), 1),         # NULL A
    ((P, 2 * P, 3 * P, 1.0, 4 * P, 8, 8, 128, 0), 2),          # ldb < N
    ((P, 2 * P, 3 * P, 1.0, 4 * P, 8, 0, 128, 16), 2),         # N = 0
    ((P, 2 * P, 3 * P, 1.0, 4 * P, 8, 9, 128, 24), 3),         # ldb % 16 != 0
    ((P, 2 * P, 3 * P, 1.0, 4 * P, 8, 9, 192, 16), 3),         # K % 128 != 0
    ((P, 2 * P + 8, 3 * P, 1.0, 4 * P, 8, 9, 128, 16), 3),     # misaligned b_t
    ((P, 2 * P, 3 * P, 1.0, 2 * P + 64, 8, 9, 128, 16), 4),    # C overlaps b_t
])
def test_w4a16_t_rejects_bad_arguments(lib, args, expect):
    f = lib.gemm_w4a16_t
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_float, ctypes.c_void_p] + [ctypes.c_int] * 4 + \
        [ctypes.c_void_p]
    assert f(*args, None) == expect


def test_testing_overrides_reject_bad_values(lib):
    f = lib.gemm_testing_set_overrides
    f.argtypes = [ctypes.c_int, ctypes.c_int]
    assert f(3, 0) == 2 and f(0, -1) == 2
    assert f(0, 0) == 0
