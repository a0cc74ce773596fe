"""Builds libgb300gemm.so in-tree with nvcc for sm_103a (one -gencode).

Each .cu in csrc/ is compiled to an object in parallel, then the objects are
linked into a shared library next to this file.  The measurement tool in
probe/ (tensor-pipe issue rate, used by bench.py --tensor-rate) is linked
into libgb300probe.so beside it.  The build is skipped when
the library is newer than every source and header.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
PROBE = os.path.join(PKG, "probe")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(ROOT, "_build", "gb300gemm")
LIB = os.path.join(PKG, "libgb300gemm.so")
# measurement tool (tensor-pipe issue rate), kept out of the GEMM library
PROBE_LIB = os.path.join(PKG, "libgb300probe.so")

GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", INCLUDE, "-I", CSRC,
]
# Per-file extra flags: the router's arithmetic must never be contracted.
EXTRA = {"gemm_router.cu": ["-fmad=false"]}


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgb300gemm.so")


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(PROBE, f) for f in os.listdir(PROBE)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(PROBE_LIB)):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(PROBE_LIB))
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(nvcc: str, src: str, verbose_ptxas: bool) -> str:
    """src: a file name in csrc/, or 'probe/<name>' for the measurement tool."""
    path = os.path.join(PKG, src) if src.startswith("probe/") else os.path.join(CSRC, src)
    obj = os.path.join(OBJDIR, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc, *GENCODE, *NVCC_FLAGS, *EXTRA.get(src, [])]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    cmd += ["-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile and link the library; returns its path."""
    if not force and not verbose_ptxas and up_to_date():
        return LIB
    nvcc = nvcc_path()
    os.makedirs(OBJDIR, exist_ok=True)
    srcs = sources()
    probes = ["probe/" + f for f in sorted(os.listdir(PROBE)) if f.endswith(".cu")]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs) + len(probes),
                                                      os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, verbose_ptxas), srcs + probes))
    for lib, parts in ((LIB, objs[:len(srcs)]), (PROBE_LIB, objs[len(srcs):])):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *GENCODE, "-shared", "-cudart", "static", "-o", tmp, *parts]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)
