"""CPU oracle for the dense NT GEMM family (TEST INFRASTRUCTURE ONLY).

Only the tests, the package smoke check and the CPU-baseline leg of
``bench.py`` may import this module.  The product library never imports it,
and it never imports the product: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, built with
``-ffp-contract=off``); this module compiles it and marshals numpy arrays.
Each wrapper names the passage it follows:

* ``gemm_bf16_nt``            - "sm121a_matmul.py" ``_sm121a_matmul_kernel``
  (FP32 accumulator, BF16 store) with the NT layout of "gemm_dense.rs"
  ``dense_gemm_tc``.
* ``gemm_bf16_nt_scaled_acc`` - "gemm_dense.rs" ``dense_gemm_tc_scaled_acc``.
* ``bf16_scaled_add``         - the second kernel of the unfused pair that the
  same docstring describes.
* ``gemm_router``             - "gemm_dense.rs" ``dense_gemm_router`` /
  ``dense_gemm`` (strict k order, no FMA).
* ``gemm_nvfp4_bs``           - "kernelbot nvfp4 gemm submission 123329",
  sections "SCALE FACTORS", "NVIDIA Block layout", "Layout semantics" and
  ``custom_kernel``.
* ``gemm_w4a16``              - "gemm_dense.rs" ``w4a16_gemm`` and its BF16
  variant ``w4a16_gemm_n128_m128_bf16`` (NVFP4 weights dequantised to BF16,
  FP32 accumulation); the layout and rounding readings are in ``oracle.c``.

Parity pins for every function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-pthread", "-Wall", "-fvisibility=hidden"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB names another build of oracle.c to load instead (the
            # planted-mistake tests load deliberately broken copies this way)
            path = os.environ.get("ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            L, I, F = ctypes.c_long, ctypes.c_int, ctypes.c_float
            lib.oracle_bf16_to_f32.restype = ctypes.c_float
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
            lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.oracle_f64_to_f16.restype = ctypes.c_uint16
            lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_e2m1_decode.restype = ctypes.c_double
            lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint]
            lib.oracle_sf_offset.restype = ctypes.c_long
            lib.oracle_sf_offset.argtypes = [L, L, L, L, L]
            lib.oracle_gemm_bf16_nt.restype = I
            lib.oracle_gemm_bf16_nt.argtypes = [u16p, u16p, u16p, L, L, L, lp, L, I]
            lib.oracle_gemm_bf16_nt_scaled_acc.restype = I
            lib.oracle_gemm_bf16_nt_scaled_acc.argtypes = [u16p, u16p, u16p, L, L, L, F, lp, L, I]
            lib.oracle_gemm_router.restype = I
            lib.oracle_gemm_router.argtypes = [u16p, u16p, f32p, L, L, L, lp, L, I]
            lib.oracle_bf16_scaled_add.restype = None
            lib.oracle_bf16_scaled_add.argtypes = [u16p, u16p, F, L]
            lib.oracle_f32_to_bf16_array.restype = None
            lib.oracle_f32_to_bf16_array.argtypes = [f32p, u16p, L]
            lib.oracle_f64_to_f16_array.restype = None
            lib.oracle_f64_to_f16_array.argtypes = [f64p, u16p, L]
            lib.oracle_gemm_nvfp4_bs.restype = I
            lib.oracle_gemm_nvfp4_bs.argtypes = [u8p, u8p, u8p, u8p, u16p, L, L, L, L, lp, L, I]
            lib.oracle_gemm_w4a16.restype = I
            lib.oracle_gemm_w4a16.argtypes = [u16p, u8p, u8p, F, u16p, L, L, L, lp, L, I]
            lib.oracle_gemm_w4a16_t.restype = I
            lib.oracle_gemm_w4a16_t.argtypes = [u16p, u8p, u8p, F, u16p, L, L, L, L, lp, L, I]
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _rows_arg(rows, total):
    if rows is None:
        return None, total, None
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return _ptr(r, ctypes.c_long), len(r), r  # keep r alive


def _u16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, "bf16/fp16 data is passed as raw uint16 bit patterns"
    return x


# --- scalar codecs ---------------------------------------------------------

def bf16_to_f32(bits: int) -> float:
    return _load().oracle_bf16_to_f32(bits)


def f32_to_bf16(x: float) -> int:
    return _load().oracle_f32_to_bf16(x)


def f64_to_f16(x: float) -> int:
    return _load().oracle_f64_to_f16(x)


def f16_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(bits)


def e2m1_decode(code: int) -> float:
    return _load().oracle_e2m1_decode(code)


def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(code)


def sf_offset(r: int, j: int, l: int, rest_rows: int, rest_k: int) -> int:
    return _load().oracle_sf_offset(r, j, l, rest_rows, rest_k)


def f32_to_bf16_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f32_to_bf16_array(_ptr(x, ctypes.c_float), _ptr(y, ctypes.c_uint16), x.size)
    return y


def f64_to_f16_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f64_to_f16_array(_ptr(x, ctypes.c_double), _ptr(y, ctypes.c_uint16), x.size)
    return y


# --- GEMMs -----------------------------------------------------------------

def gemm_bf16_nt(A: np.ndarray, B: np.ndarray, rows=None, threads: int | None = None) -> np.ndarray:
    """C[rows] = bf16(fp32-sequential A[rows] @ B^T); A [M,K], B [N,K] as uint16 bf16 bits."""
    A, B = _u16(A), _u16(B)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    rp, nrows, _keep = _rows_arg(rows, M)
    C = np.empty((nrows, N), dtype=np.uint16)
    rc = _load().oracle_gemm_bf16_nt(_ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16),
                                     _ptr(C, ctypes.c_uint16), M, N, K, rp, nrows,
                                     threads or default_threads())
    assert rc == 0, f"oracle_gemm_bf16_nt rc={rc}"
    return C


def gemm_bf16_nt_scaled_acc(A, B, out_init, scale: float, rows=None, threads=None) -> np.ndarray:
    """out[rows] = bf16(out + scale*bf16(A[rows] @ B^T)); out_init holds those rows' initial values."""
    A, B = _u16(A), _u16(B)
    M, K = A.shape
    N, _ = B.shape
    rp, nrows, _keep = _rows_arg(rows, M)
    out = np.array(_u16(out_init), copy=True).reshape(nrows, N)
    rc = _load().oracle_gemm_bf16_nt_scaled_acc(_ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16),
                                                _ptr(out, ctypes.c_uint16), M, N, K,
                                                float(scale), rp, nrows, threads or default_threads())
    assert rc == 0, f"oracle_gemm_bf16_nt_scaled_acc rc={rc}"
    return out


def bf16_scaled_add(out: np.ndarray, d: np.ndarray, scale: float) -> np.ndarray:
    """Return bf16(out + scale*d) elementwise (the unfused pair's second step)."""
    o = np.array(_u16(out), copy=True)
    dd = _u16(d)
    assert o.size == dd.size
    _load().oracle_bf16_scaled_add(_ptr(o, ctypes.c_uint16), _ptr(dd, ctypes.c_uint16), float(scale), o.size)
    return o


def gemm_router(A, B, rows=None, threads=None) -> np.ndarray:
    """FP32 C[rows] = strict-order, FMA-free sum_k A[m,k]*B[n,k]."""
    A, B = _u16(A), _u16(B)
    M, K = A.shape
    N, _ = B.shape
    rp, nrows, _keep = _rows_arg(rows, M)
    C = np.empty((nrows, N), dtype=np.float32)
    rc = _load().oracle_gemm_router(_ptr(A, ctypes.c_uint16), _ptr(B, ctypes.c_uint16),
                                    _ptr(C, ctypes.c_float), M, N, K, rp, nrows,
                                    threads or default_threads())
    assert rc == 0, f"oracle_gemm_router rc={rc}"
    return C


def gemm_nvfp4_bs(a: np.ndarray, b: np.ndarray, sfa: np.ndarray, sfb: np.ndarray,
                  L: int, M: int, N: int, K: int, rows=None, threads=None) -> np.ndarray:
    """fp16 bits of c[rows] for the NVFP4 block-scaled GEMM; rows are flat l*M+m ids.

    a: uint8 [L,M,K/2], b: uint8 [L,N,K/2], sfa/sfb: uint8 in the hardware
    scale layout (L*M*K/16 and L*N*K/16 bytes).
    """
    a = np.ascontiguousarray(a, dtype=np.uint8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    sfa = np.ascontiguousarray(sfa, dtype=np.uint8)
    sfb = np.ascontiguousarray(sfb, dtype=np.uint8)
    assert a.size == L * M * K // 2 and b.size == L * N * K // 2
    assert sfa.size == L * M * K // 16 and sfb.size == L * N * K // 16
    rp, nrows, _keep = _rows_arg(rows, L * M)
    C = np.empty((nrows, N), dtype=np.uint16)
    rc = _load().oracle_gemm_nvfp4_bs(_ptr(a, ctypes.c_uint8), _ptr(b, ctypes.c_uint8),
                                      _ptr(sfa, ctypes.c_uint8), _ptr(sfb, ctypes.c_uint8),
                                      _ptr(C, ctypes.c_uint16), L, M, N, K, rp, nrows,
                                      threads or default_threads())
    assert rc == 0, f"oracle_gemm_nvfp4_bs rc={rc}"
    return C


def gemm_w4a16(A: np.ndarray, b: np.ndarray, sfb: np.ndarray, scale2: float, rows=None,
               threads=None) -> np.ndarray:
    """bf16 bits of C[rows] = bf16(scale2 * fp32-sequential A[rows] @ w^T) with
    the exact block-scaled weights w[n,k] = e2m1(b[n,k]) * e4m3(sfb[n,k/16]).

    A: uint16 bf16 bits [M,K]; b: uint8 [N,K/2] (low nibble = even k);
    sfb: uint8 e4m3 [N,K/16]; scale2: the FP32 per-tensor scale.
    """
    A = _u16(A)
    M, K = A.shape
    b = np.ascontiguousarray(b, dtype=np.uint8)
    sfb = np.ascontiguousarray(sfb, dtype=np.uint8)
    N = b.shape[0]
    assert b.size == N * K // 2 and sfb.size == N * K // 16
    rp, nrows, _keep = _rows_arg(rows, M)
    C = np.empty((nrows, N), dtype=np.uint16)
    rc = _load().oracle_gemm_w4a16(_ptr(A, ctypes.c_uint16), _ptr(b, ctypes.c_uint8),
                                   _ptr(sfb, ctypes.c_uint8), float(np.float32(scale2)),
                                   _ptr(C, ctypes.c_uint16), M, N, K, rp, nrows,
                                   threads or default_threads())
    assert rc == 0, f"oracle_gemm_w4a16 rc={rc}"
    return C



def gemm_w4a16_t(A: np.ndarray, b_t: np.ndarray, sfb_t: np.ndarray, scale2: float, N: int,
                 rows=None, threads=None) -> np.ndarray:
    """gemm_w4a16 with the weights in the transposed layout.

    b_t: uint8 [K/2, ldb], byte (j, n) = elements 2j (low nibble) and 2j+1
    (high nibble) of weight column n; sfb_t: uint8 e4m3 [K/16, ldb], byte
    (j, n) scaling elements 16j..16j+15 of column n; columns n >= N are
    padding and never read.
    """
    A = _u16(A)
    M, K = A.shape
    b_t = np.ascontiguousarray(b_t, dtype=np.uint8)
    sfb_t = np.ascontiguousarray(sfb_t, dtype=np.uint8)
    ldb = b_t.shape[1]
    assert b_t.shape == (K // 2, ldb) and sfb_t.shape == (K // 16, ldb) and ldb >= N
    rp, nrows, _keep = _rows_arg(rows, M)
    C = np.empty((nrows, N), dtype=np.uint16)
    rc = _load().oracle_gemm_w4a16_t(_ptr(A, ctypes.c_uint16), _ptr(b_t, ctypes.c_uint8),
                                     _ptr(sfb_t, ctypes.c_uint8), float(np.float32(scale2)),
                                     _ptr(C, ctypes.c_uint16), M, N, K, ldb, rp, nrows,
                                     threads or default_threads())
    assert rc == 0, f"oracle_gemm_w4a16_t rc={rc}"
    return C
