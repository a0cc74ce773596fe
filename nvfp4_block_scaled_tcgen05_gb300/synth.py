"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and lays them out as raw bit patterns
(uint16 for bf16, uint8 for packed e2m1 and e4m3 scale bytes).  It holds none
of the GEMM arithmetic and imports neither the CUDA binding nor the oracle.

Workloads (shapes and value distributions from the pages' target shapes: the
Qwen-2B-shaped LoRA-training GEMMs of "sm121a_matmul.py", the LoRA fold
width n = 17408 and the router shapes of "gemm_dense.rs", and the NVFP4
problem sizes of the kernelbot submission):

* ``tiny``    A[128,256], B[256,256] ~ N(0,1); out[128,256] ~ N(0,1), scale 0.5
* ``gateup``  M=5120 N=11008 K=2048, A ~ N(0,1), B ~ N(0,0.02)
* ``down``    M=5120 N=2048  K=11008
* ``qkv``     M=5120 N=2048  K=2048
* ``gqa``     M=5120 N=512   K=2048
* ``lora``    out[4096,17408] ~ N(0,1) += 2.0 * bf16(X[4096,16] ~ N(0,1) . W[17408,16] ~ N(0,0.01)^T)
* ``router``  A[4510,2048], B[256,2048] ~ N(0,1) -> FP32
* ``nvfp4``   L=1 M=4096 N=7168 K=16384; e2m1 codes uniform over all 16
  values (uniform bytes), scales 2^U{-4..2} stored as e4m3 bytes.
* ``w4a16_qkvz`` A[1016,2048] ~ N(0,1) bf16 times NVFP4 weights [12288,2048]
  (the qkvz projection at ISL 1016 of "gemm_dense.rs" w4a16_gemm_n128_m128):
  e2m1 codes uniform, e4m3 block scales uniform over the codes of
  2^-4 .. 2^2 (mantissas included), per-tensor scale 0.0123.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

# e4m3 bit patterns of the powers of two 2^-4 .. 2^2 (sign 0, exponent field
# e+7, mantissa 0).  Scales are i.i.d., so their placement in the hardware
# layout needs no index arithmetic here: every byte of the buffer is drawn.
E4M3_POW2_BYTES = {-4: 0x18, -3: 0x20, -2: 0x28, -1: 0x30, 0: 0x38, 1: 0x40, 2: 0x48}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def bf16_normal(shape, sigma: float, seed: int) -> np.ndarray:
    """N(0, sigma^2) samples cast to bf16 (round to nearest even); returns uint16 bits."""
    g = _gen(seed)
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if sigma != 1.0:
        x = x * sigma
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_small_ints(shape, lo: int, hi: int, seed: int) -> np.ndarray:
    """Integers uniform in [lo, hi] as bf16 bits (exactly representable)."""
    g = _gen(seed)
    x = torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int32).to(torch.float32)
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def uniform_bytes(n: int, seed: int) -> np.ndarray:
    """n uniform random bytes (= two uniform e2m1 codes per byte)."""
    g = _gen(seed)
    return torch.randint(0, 256, (int(n),), generator=g, dtype=torch.int32).to(torch.uint8).numpy()


def pow2_scale_bytes(n: int, seed: int, lo: int = -4, hi: int = 2) -> np.ndarray:
    """n e4m3 scale bytes, each 2^e with e uniform in [lo, hi]."""
    g = _gen(seed)
    e = torch.randint(lo, hi + 1, (int(n),), generator=g, dtype=torch.int32).numpy()
    table = np.zeros(hi - lo + 1, dtype=np.uint8)
    for k in range(lo, hi + 1):
        table[k - lo] = E4M3_POW2_BYTES[k]
    return table[e - lo]


@dataclass(frozen=True)
class Gemm:
    name: str
    M: int
    N: int
    K: int
    sigma_a: float = 1.0
    sigma_b: float = 1.0
    seed: int = 1000


BF16_WORKLOADS = {
    "tiny": Gemm("tiny", 128, 256, 256, 1.0, 1.0, 1000),
    "gateup": Gemm("gateup", 5120, 11008, 2048, 1.0, 0.02, 1001),
    "down": Gemm("down", 5120, 2048, 11008, 1.0, 0.02, 1002),
    "qkv": Gemm("qkv", 5120, 2048, 2048, 1.0, 0.02, 1012),
    "gqa": Gemm("gqa", 5120, 512, 2048, 1.0, 0.02, 1022),
}
LORA = Gemm("lora", 4096, 17408, 16, 1.0, 0.01, 1003)
LORA_SCALE = 2.0
TINY_SCALE = 0.5
ROUTER = Gemm("router", 4510, 256, 2048, 1.0, 1.0, 1013)


@dataclass(frozen=True)
class Nvfp4:
    name: str
    L: int
    M: int
    N: int
    K: int
    seed: int = 1004


NVFP4 = Nvfp4("nvfp4", 1, 4096, 7168, 16384, 1004)
# decode-like shapes of the NVFP4 page's benchmark (M = 128) and their K
# split counts: the swapped kernel puts 256 weight rows on a CTA pair, so
# (N / 256) x splits work units share 76 pairs: 56 units at 7168 x 16384
# (2 splits), 64 at 4096 x 7168 (4 splits), the fastest counts measured
# (more splits give each unit too few K blocks to amortise its start-up
# and its transposed partial stores)
NVFP4_DECODE = {
    "nvfp4_decode_7168x16384": (Nvfp4("nvfp4_decode_7168x16384", 1, 128, 7168, 16384, 1005), 2),
    "nvfp4_decode_4096x7168": (Nvfp4("nvfp4_decode_4096x7168", 1, 128, 4096, 7168, 1006), 4),
}


def gemm_inputs(w: Gemm, seed_offset: int = 0):
    """(A [M,K], B [N,K]) bf16 bits for a BF16 workload."""
    A = bf16_normal((w.M, w.K), w.sigma_a, w.seed + 17 * seed_offset)
    B = bf16_normal((w.N, w.K), w.sigma_b, w.seed + 17 * seed_offset + 1)
    return A, B


def scaled_acc_out(M: int, N: int, seed: int) -> np.ndarray:
    """Initial values of the accumulated output, ~ N(0,1) bf16 bits."""
    return bf16_normal((M, N), 1.0, seed + 2)


def e4m3_range_bytes(n: int, seed: int, lo: int = 0x18, hi: int = 0x48) -> np.ndarray:
    """n e4m3 scale bytes uniform over the codes lo..hi (positive normals)."""
    g = _gen(seed)
    return torch.randint(lo, hi + 1, (int(n),), generator=g, dtype=torch.int32).to(torch.uint8).numpy()


@dataclass(frozen=True)
class W4a16:
    name: str
    M: int
    N: int
    K: int
    scale2: float = 0.0123
    seed: int = 1007


W4A16 = {
    "w4a16_qkvz": W4a16("w4a16_qkvz", 1016, 12288, 2048),
}


def w4a16_inputs(w: W4a16, seed_offset: int = 0):
    """(A [M,K] bf16 bits, b [N,K/2] packed e2m1, sfb [N,K/16] e4m3 bytes, scale2)."""
    s = w.seed + 17 * seed_offset
    A = bf16_normal((w.M, w.K), 1.0, s)
    b = uniform_bytes(w.N * w.K // 2, s + 1).reshape(w.N, w.K // 2)
    sfb = e4m3_range_bytes(w.N * w.K // 16, s + 2).reshape(w.N, w.K // 16)
    return A, b, sfb, float(np.float32(w.scale2))


def nvfp4_inputs(w: Nvfp4, seed_offset: int = 0):
    """(a [L,M,K/2], b [L,N,K/2], sfa, sfb) as uint8; scale buffers are flat."""
    s = w.seed + 17 * seed_offset
    a = uniform_bytes(w.L * w.M * w.K // 2, s).reshape(w.L, w.M, w.K // 2)
    b = uniform_bytes(w.L * w.N * w.K // 2, s + 1).reshape(w.L, w.N, w.K // 2)
    sfa = pow2_scale_bytes(w.L * w.M * w.K // 16, s + 2)
    sfb = pow2_scale_bytes(w.L * w.N * w.K // 16, s + 3)
    return a, b, sfa, sfb
