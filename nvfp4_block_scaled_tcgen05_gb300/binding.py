"""Thin Python binding over the C ABI in include/gb300gemm.h.

Argument marshalling only: every function checks dtypes/shapes/devices of
the torch tensors it is given, passes their device pointers and the current
CUDA stream to the C entry point of the same name, and raises GemmError on
a non-zero status.  All arithmetic runs in the library's CUDA kernels; there
is no fallback path.  A missing library raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

STATUS = {
    0: "GEMM_OK", 1: "GEMM_ERR_NULL", 2: "GEMM_ERR_SHAPE", 3: "GEMM_ERR_ALIGN",
    4: "GEMM_ERR_ALIAS", 5: "GEMM_ERR_ARCH", 6: "GEMM_ERR_LAUNCH", 7: "GEMM_ERR_TIMEOUT",
    8: "GEMM_ERR_NO_DEVICE", 9: "GEMM_ERR_CAPTURE",
}
EXPORTS = ("gemm_bf16_nt", "gemm_bf16_nn", "gemm_bf16_nt_scaled_acc", "gemm_bf16_nt_ordered", "gemm_nvfp4_bs",
           "gemm_bf16_nt_splitk", "gemm_bf16_nt_streamk", "gemm_nvfp4_bs_splitk", "gemm_w4a16", "gemm_w4a16_t", "gemm_w4a16_ws",
           "bf16_scaled_add", "gemm_get_device_status", "gemm_selftest_wait_timeout",
           "gemm_testing_set_overrides", "gemm_status_string")


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libgb300gemm.so (built in-tree); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(path)
            vp, i, f, l = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_long
            lib.gemm_bf16_nt.argtypes = [vp, vp, vp, i, i, i, vp]
            lib.gemm_bf16_nn.argtypes = [vp, vp, vp, i, i, i, vp]
            lib.gemm_bf16_nt_scaled_acc.argtypes = [vp, vp, vp, i, i, i, f, vp]
            lib.gemm_bf16_nt_ordered.argtypes = [vp, vp, vp, i, i, i, vp]
            lib.gemm_nvfp4_bs.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
            lib.bf16_scaled_add.argtypes = [vp, vp, f, l, vp]
            lib.gemm_bf16_nt_splitk.argtypes = [vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, vp]
            lib.gemm_bf16_nt_splitk_workspace_bytes.argtypes = [i, i, i, i]
            lib.gemm_bf16_nt_splitk_workspace_bytes.restype = ctypes.c_size_t
            lib.gemm_bf16_nt_streamk.argtypes = [vp, vp, vp, vp, ctypes.c_size_t, i, i, i, vp]
            lib.gemm_w4a16.argtypes = [vp, vp, vp, f, vp, i, i, i, vp]
            lib.gemm_w4a16_t.argtypes = [vp, vp, vp, f, vp, i, i, i, i, vp]
            lib.gemm_w4a16_ws.argtypes = [vp, vp, vp, f, vp, vp, ctypes.c_size_t, i, i, i, vp]
            lib.gemm_w4a16_ws_workspace_bytes.argtypes = [i, i]
            lib.gemm_w4a16_ws_workspace_bytes.restype = ctypes.c_size_t
            lib.gemm_bf16_nt_streamk_workspace_bytes.argtypes = []
            lib.gemm_bf16_nt_streamk_workspace_bytes.restype = ctypes.c_size_t
            lib.gemm_nvfp4_bs_splitk.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                                 i, i, i, i, i, vp]
            lib.gemm_nvfp4_bs_splitk_workspace_bytes.argtypes = [i, i, i, i]
            lib.gemm_nvfp4_bs_splitk_workspace_bytes.restype = ctypes.c_size_t
            lib.gemm_get_device_status.argtypes = [vp]
            lib.gemm_selftest_wait_timeout.argtypes = [i, vp]
            lib.gemm_testing_set_overrides.argtypes = [i, i]
            lib.gemm_status_string.argtypes = [i]
            lib.gemm_status_string.restype = ctypes.c_char_p
            for name in EXPORTS[:-1]:
                getattr(lib, name).restype = i
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    try:
        return load().gemm_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS.get(int(status), "unknown status")


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise GemmError(rc, where)


def _mat(t: torch.Tensor, dtype, name: str, ndim: int = 2) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (row-major)")


def gemm_bf16_nt(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, stream=None):
    """C[M,N] = bf16(A[M,K] . B[N,K]^T), FP32 accumulation on tcgen05 tensor cores."""
    _mat(A, torch.bfloat16, "A")
    _mat(B, torch.bfloat16, "B")
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError(f"K mismatch: A {tuple(A.shape)} vs B {tuple(B.shape)}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _mat(C, torch.bfloat16, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError("C must be [M, N]")
    _check(load().gemm_bf16_nt(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                               _stream_ptr(stream)), "gemm_bf16_nt")
    return C


def gemm_bf16_nn(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, stream=None):
    """C[M,N] = bf16(A[M,K] . B[K,N]) (B row-major [K][N]), FP32 accumulation."""
    _mat(A, torch.bfloat16, "A")
    _mat(B, torch.bfloat16, "B")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"K mismatch: A {tuple(A.shape)} vs B {tuple(B.shape)}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _mat(C, torch.bfloat16, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError("C must be [M, N]")
    _check(load().gemm_bf16_nn(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                               _stream_ptr(stream)), "gemm_bf16_nn")
    return C


def gemm_bf16_nt_scaled_acc(A: torch.Tensor, B: torch.Tensor, C_inout: torch.Tensor, scale: float,
                            stream=None):
    """C_inout = bf16(C_inout + scale * bf16(A . B^T)) in place (fused LoRA fold)."""
    _mat(A, torch.bfloat16, "A")
    _mat(B, torch.bfloat16, "B")
    _mat(C_inout, torch.bfloat16, "C_inout")
    M, K = A.shape
    N, _ = B.shape
    if tuple(C_inout.shape) != (M, N) or B.shape[1] != K:
        raise ValueError("shape mismatch")
    _check(load().gemm_bf16_nt_scaled_acc(A.data_ptr(), B.data_ptr(), C_inout.data_ptr(), M, N, K,
                                          float(scale), _stream_ptr(stream)),
           "gemm_bf16_nt_scaled_acc")
    return C_inout


def gemm_bf16_nt_splitk_workspace_bytes(M: int, N: int, K: int, k_splits: int) -> int:
    return int(load().gemm_bf16_nt_splitk_workspace_bytes(M, N, K, k_splits))


def gemm_bf16_nt_splitk(A: torch.Tensor, B: torch.Tensor, k_splits: int,
                        workspace: torch.Tensor | None = None, C: torch.Tensor | None = None,
                        stream=None):
    """C = bf16(sum over K splits of FP32 partials), split-K with a caller workspace."""
    _mat(A, torch.bfloat16, "A")
    _mat(B, torch.bfloat16, "B")
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("K mismatch")
    need = gemm_bf16_nt_splitk_workspace_bytes(M, N, K, k_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=A.device)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _mat(C, torch.bfloat16, "C")
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().gemm_bf16_nt_splitk(A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                      workspace.data_ptr(), nbytes, M, N, K, int(k_splits),
                                      _stream_ptr(stream)), "gemm_bf16_nt_splitk")
    return C


def gemm_bf16_nt_streamk_workspace_bytes() -> int:
    return int(load().gemm_bf16_nt_streamk_workspace_bytes())


def gemm_bf16_nt_streamk(A: torch.Tensor, B: torch.Tensor, workspace: torch.Tensor | None = None,
                         C: torch.Tensor | None = None, stream=None):
    """C = bf16(A . B^T) on the stream-K schedule, with a caller workspace."""
    _mat(A, torch.bfloat16, "A")
    _mat(B, torch.bfloat16, "B")
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("K mismatch")
    if workspace is None:
        need = gemm_bf16_nt_streamk_workspace_bytes()
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=A.device)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _mat(C, torch.bfloat16, "C")
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().gemm_bf16_nt_streamk(A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                       workspace.data_ptr(), nbytes, M, N, K,
                                       _stream_ptr(stream)), "gemm_bf16_nt_streamk")
    return C


def gemm_w4a16(A: torch.Tensor, b: torch.Tensor, sfb: torch.Tensor, scale2: float,
               C: torch.Tensor | None = None, stream=None):
    """C = bf16(scale2 * (A . w^T)), w = e2m1(b) * e4m3(sfb) (exact in bf16).

    A bf16 [M,K]; b uint8 [N,K/2] packed e2m1 (low nibble = even k);
    sfb uint8 [N,K/16] e4m3 block scales; C bf16 [M,N].
    """
    _mat(A, torch.bfloat16, "A")
    _mat(b, torch.uint8, "b")
    _mat(sfb, torch.uint8, "sfb")
    M, K = A.shape
    N = b.shape[0]
    if tuple(b.shape) != (N, K // 2) or tuple(sfb.shape) != (N, K // 16):
        raise ValueError("shape mismatch")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _mat(C, torch.bfloat16, "C")
    _check(load().gemm_w4a16(A.data_ptr(), b.data_ptr(), sfb.data_ptr(), float(scale2),
                             C.data_ptr(), M, N, K, _stream_ptr(stream)), "gemm_w4a16")
    return C


def gemm_w4a16_t(A: torch.Tensor, b_t: torch.Tensor, sfb_t: torch.Tensor, scale2: float, N: int,
                 C: torch.Tensor | None = None, stream=None):
    """gemm_w4a16 with the transposed weight layout.

    A bf16 [M,K]; b_t uint8 [K/2, ldb], byte (j, n) = elements 2j (low
    nibble) and 2j+1 (high nibble) of weight column n; sfb_t uint8 e4m3
    [K/16, ldb]; ldb >= N (columns >= N are padding); C bf16 [M,N].
    """
    _mat(A, torch.bfloat16, "A")
    _mat(b_t, torch.uint8, "b_t")
    _mat(sfb_t, torch.uint8, "sfb_t")
    M, K = A.shape
    ldb = b_t.shape[1]
    if tuple(b_t.shape) != (K // 2, ldb) or tuple(sfb_t.shape) != (K // 16, ldb):
        raise ValueError("shape mismatch")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _mat(C, torch.bfloat16, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError("C must be [M, N]")
    _check(load().gemm_w4a16_t(A.data_ptr(), b_t.data_ptr(), sfb_t.data_ptr(), float(scale2),
                               C.data_ptr(), M, N, K, ldb, _stream_ptr(stream)), "gemm_w4a16_t")
    return C


def gemm_w4a16_ws_workspace_bytes(N: int, K: int) -> int:
    return int(load().gemm_w4a16_ws_workspace_bytes(N, K))


def gemm_w4a16_ws(A: torch.Tensor, b: torch.Tensor, sfb: torch.Tensor, scale2: float,
                  workspace: torch.Tensor | None = None, C: torch.Tensor | None = None,
                  stream=None):
    """gemm_w4a16 in two passes (weights converted once into the workspace)."""
    _mat(A, torch.bfloat16, "A")
    _mat(b, torch.uint8, "b")
    _mat(sfb, torch.uint8, "sfb")
    M, K = A.shape
    N = b.shape[0]
    if tuple(b.shape) != (N, K // 2) or tuple(sfb.shape) != (N, K // 16):
        raise ValueError("shape mismatch")
    if workspace is None:
        workspace = torch.empty(max(gemm_w4a16_ws_workspace_bytes(N, K), 16), dtype=torch.uint8,
                                device=A.device)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _mat(C, torch.bfloat16, "C")
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().gemm_w4a16_ws(A.data_ptr(), b.data_ptr(), sfb.data_ptr(), float(scale2),
                                C.data_ptr(), workspace.data_ptr(), nbytes, M, N, K,
                                _stream_ptr(stream)), "gemm_w4a16_ws")
    return C


def gemm_bf16_nt_ordered(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None,
                         stream=None):
    """FP32 C = strict-order, FMA-free A . B^T on CUDA cores (router GEMM)."""
    _mat(A, torch.bfloat16, "A")
    _mat(B, torch.bfloat16, "B")
    M, K = A.shape
    N, _ = B.shape
    if B.shape[1] != K:
        raise ValueError("K mismatch")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _mat(C, torch.float32, "C")
    _check(load().gemm_bf16_nt_ordered(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                       _stream_ptr(stream)), "gemm_bf16_nt_ordered")
    return C


def gemm_nvfp4_bs(a: torch.Tensor, b: torch.Tensor, sfa: torch.Tensor, sfb: torch.Tensor,
                  L: int, M: int, N: int, K: int, c: torch.Tensor | None = None, stream=None):
    """fp16 c[L,M,N] for packed-e2m1 a[L,M,K/2], b[L,N,K/2] (uint8) with e4m3 scale
    bytes sfa (L*M*K/16), sfb (L*N*K/16) in the hardware scale layout."""
    for t, n in ((a, "a"), (b, "b"), (sfa, "sfa"), (sfb, "sfb")):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{n} must be a contiguous CUDA uint8 tensor")
    if a.numel() != L * M * K // 2 or b.numel() != L * N * K // 2:
        raise ValueError("a/b size mismatch")
    if sfa.numel() != L * M * K // 16 or sfb.numel() != L * N * K // 16:
        raise ValueError("scale buffer size mismatch")
    if c is None:
        c = torch.empty((L, M, N), dtype=torch.float16, device=a.device)
    if c.dtype != torch.float16 or not c.is_contiguous() or c.numel() != L * M * N:
        raise ValueError("c must be a contiguous fp16 [L, M, N] tensor")
    _check(load().gemm_nvfp4_bs(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                                c.data_ptr(), L, M, N, K, _stream_ptr(stream)), "gemm_nvfp4_bs")
    return c


def gemm_nvfp4_bs_splitk_workspace_bytes(M: int, N: int, K: int, k_splits: int) -> int:
    return int(load().gemm_nvfp4_bs_splitk_workspace_bytes(M, N, K, k_splits))


def gemm_nvfp4_bs_splitk(a: torch.Tensor, b: torch.Tensor, sfa: torch.Tensor, sfb: torch.Tensor,
                         M: int, N: int, K: int, k_splits: int,
                         workspace: torch.Tensor | None = None, c: torch.Tensor | None = None,
                         stream=None, L: int = 1):
    """fp16 c[L,M,N] = gemm_nvfp4_bs with K split into k_splits chunks."""
    for t, n in ((a, "a"), (b, "b"), (sfa, "sfa"), (sfb, "sfb")):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{n} must be a contiguous CUDA uint8 tensor")
    if a.numel() != L * M * K // 2 or b.numel() != L * N * K // 2:
        raise ValueError("a/b size mismatch")
    if sfa.numel() != L * M * K // 16 or sfb.numel() != L * N * K // 16:
        raise ValueError("scale buffer size mismatch")
    need = L * gemm_nvfp4_bs_splitk_workspace_bytes(M, N, K, k_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=a.device)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if c is None:
        c = torch.empty((L, M, N), dtype=torch.float16, device=a.device)
    if c.dtype != torch.float16 or not c.is_contiguous() or c.numel() != L * M * N:
        raise ValueError("c must be a contiguous fp16 [L, M, N] tensor")
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().gemm_nvfp4_bs_splitk(a.data_ptr(), b.data_ptr(), sfa.data_ptr(), sfb.data_ptr(),
                                       c.data_ptr(), workspace.data_ptr(), nbytes, L, M, N, K,
                                       int(k_splits), _stream_ptr(stream)), "gemm_nvfp4_bs_splitk")
    return c


def bf16_scaled_add(out: torch.Tensor, d: torch.Tensor, scale: float, stream=None):
    """out = bf16(out + scale * d) elementwise (the unfused pair's second step)."""
    if out.dtype != torch.bfloat16 or d.dtype != torch.bfloat16 or out.numel() != d.numel():
        raise ValueError("out and d must be bf16 tensors of the same size")
    if not (out.is_cuda and d.is_cuda and out.is_contiguous() and d.is_contiguous()):
        raise ValueError("out and d must be contiguous CUDA tensors")
    _check(load().bf16_scaled_add(out.data_ptr(), d.data_ptr(), float(scale), out.numel(),
                                  _stream_ptr(stream)), "bf16_scaled_add")
    return out


def gemm_selftest_wait_timeout(timeout_ms: int = 50, stream=None) -> None:
    """Launch the failure-path self test (a wait that must run out)."""
    _check(load().gemm_selftest_wait_timeout(int(timeout_ms), _stream_ptr(stream)),
           "gemm_selftest_wait_timeout")


def gemm_testing_set_overrides(cta_group: int = 0, streamk_clusters: int = 0) -> None:
    """Testing hook: force the CTA group of the BF16 launchers (1 or 2) and the
    CTA pairs sharing a stream-K tail; 0 restores the shape's own choice."""
    _check(load().gemm_testing_set_overrides(int(cta_group), int(streamk_clusters)),
           "gemm_testing_set_overrides")


def gemm_get_device_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status word."""
    return int(load().gemm_get_device_status(_stream_ptr(stream)))
