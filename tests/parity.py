"""Comparison rules shared by the GPU parity tests.

* bit-exact where the method fixes the result (router, exact-integer inputs,
  fused vs unfused scaled-acc);
* otherwise every element within 1 ULP of the oracle's rounded value
  (ordered-bits distance <= 1, +0 and -0 equal) OR |diff| <= 1e-5*K*max|a|*max|b|;
* a non-finite value passes only if the oracle has the same one.
"""
from __future__ import annotations

import numpy as np
import torch


def to_dev_bf16(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).view(torch.bfloat16).to(device)


def to_dev_u8(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_val(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f16_val(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def check_close16(got: np.ndarray, ref: np.ndarray, K: int, amax: float, bmax: float,
                  fmt: str = "bf16", what: str = "") -> dict:
    """Assert the 16-bit outputs satisfy the 1-ULP-or-absolute rule; return stats."""
    got = np.asarray(got, dtype=np.uint16)
    ref = np.asarray(ref, dtype=np.uint16)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    val = bf16_val if fmt == "bf16" else f16_val
    g, r = val(got), val(ref)
    fin_r, fin_g = np.isfinite(r), np.isfinite(g)
    same_nonfinite = (~fin_r) & (~fin_g) & ((np.isnan(r) & np.isnan(g)) | (g == r))
    ulp = np.abs(_ordered(got) - _ordered(ref))
    tol = 1e-5 * K * amax * bmax
    ok = (fin_r & fin_g & ((ulp <= 1) | (np.abs(g - r) <= tol))) | same_nonfinite
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        detail = [(tuple(i), float(g[tuple(i)]), float(r[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} elements out of tolerance; "
                             f"first (index, gpu, oracle): {detail}")
    return {"max_ulp": int(ulp[fin_r & fin_g].max(initial=0)),
            "frac_exact": float((ulp == 0).mean())}


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (subnormal spacing below 2^-126)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0**-126)))
    return np.exp2(e - 7)


def check_scaled_acc(got: np.ndarray, ref_out: np.ndarray, ref_d: np.ndarray, scale: float,
                     K: int, amax: float, bmax: float, what: str = "") -> dict:
    """Scaled-acc rule.  The GEMM delta d = bf16(A.B^T) obeys the 1-ULP-or-
    absolute rule; out = bf16(o0 + scale*d) then differs from the oracle by
    at most |scale| * (d's allowance) + 1 ULP of the result (the two final
    roundings).  Exact wherever the deltas agree."""
    got = np.asarray(got, dtype=np.uint16)
    ref_out = np.asarray(ref_out, dtype=np.uint16)
    g, r, d = bf16_val(got), bf16_val(ref_out), bf16_val(ref_d)
    d_allow = np.maximum(ulp_bf16(d), 1e-5 * K * amax * bmax)
    allow = abs(scale) * d_allow + ulp_bf16(np.maximum(np.abs(g), np.abs(r)))
    fin = np.isfinite(r) & np.isfinite(g)
    ok = (fin & (np.abs(g - r) <= allow)) | (~np.isfinite(r) & ((g == r) | (np.isnan(g) & np.isnan(r))))
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        detail = [(tuple(i), float(g[tuple(i)]), float(r[tuple(i)]), float(d[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} out of tolerance; "
                             f"first (index, gpu, oracle, oracle delta): {detail}")
    ulp = np.abs(_ordered(got) - _ordered(ref_out))
    return {"max_ulp": int(ulp[fin].max(initial=0)), "frac_exact": float((ulp == 0).mean())}


def check_bitexact16(got: np.ndarray, ref: np.ndarray, what: str = "", zero_sign: bool = False):
    """Bit-exact 16-bit comparison; +0/-0 treated as equal unless zero_sign."""
    got = np.asarray(got, dtype=np.uint16)
    ref = np.asarray(ref, dtype=np.uint16)
    if zero_sign:
        eq = got == ref
    else:
        eq = (got == ref) | (((got & 0x7FFF) == 0) & ((ref & 0x7FFF) == 0))
    if not eq.all():
        idx = np.argwhere(~eq)[:5]
        raise AssertionError(f"{what}: {int((~eq).sum())} elements differ; first {idx.tolist()} "
                             f"gpu={[hex(got[tuple(i)]) for i in idx]} "
                             f"oracle={[hex(ref[tuple(i)]) for i in idx]}")


def sample_rows(M: int, tile: int = 128, n_random: int = 96, seed: int = 0) -> np.ndarray:
    """All rows of the first and last M-tile, rows around every 4th tile
    boundary, plus random rows."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(tile, M)))
    rows |= set(range(max(0, M - tile), M))
    for b in range(tile, M, 4 * tile):
        rows |= {b - 1, b, min(M - 1, b + 31), min(M - 1, b + 32)}
    rows |= set(rng.integers(0, M, size=n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)
