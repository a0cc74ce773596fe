"""The oracle's pins have teeth: each test here plants one plausible mistake
in a copy of oracle.c (a dropped k term, a fused multiply-add, a wrong
rounding tie, a wrong exponent bias, a transposed scale-layout index, a
skipped rounding of the scaled-acc delta, the wrong W4A16 scale group),
builds it, and checks that the pin suite (tests/test_oracle_pins.py) fails
against it.  The product library is not involved; everything runs on the
CPU."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# name -> (text in oracle.c, the mistake that replaces it)
MUTATIONS = {
    "dropped_last_k_term": (
        "for (long k = 0; k < K; ++k) {\n        float p = a[k] * b[k];",
        "for (long k = 0; k + 1 < K; ++k) {\n        float p = a[k] * b[k];"),
    "fused_multiply_add": (
        "float p = a[k] * b[k];\n        acc = acc + p;",
        "acc = fmaf(a[k], b[k], acc);"),
    "bf16_ties_round_up": (
        "(dropped == 0x8000u && (kept & 1u))",
        "(dropped == 0x8000u)"),
    "f16_ties_round_up": (
        "(rem == 0.5 && fmod(fl, 2.0) != 0.0)",
        "(rem == 0.5)"),
    "f16_no_subnormals": (
        "int q = (e2 >= -13) ? (e2 - 11) : -24;",
        "int q = e2 - 11;"),
    "e4m3_bias_8": (
        "else v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);",
        "else v = ldexp(1.0 + (double)m / 8.0, (int)e - 8);"),
    "e2m1_bias_0": (
        "ldexp(1.0 + 0.5 * (double)m, (int)e - 1)",
        "ldexp(1.0 + 0.5 * (double)m, (int)e)"),
    "scale_layout_g_and_i_m_swapped": (
        "+ g * 16L + i_m * 4L + i_k;",
        "+ i_m * 128L + g * 4L + i_k;"),
    "scaled_acc_delta_not_rounded": (
        "float d = oracle_bf16_to_f32(oracle_f32_to_bf16(acc));",
        "float d = acc;"),
    "w4a16_scale_per_32": (
        "sfb[n * (K / 16) + k / 16]",
        "sfb[n * (K / 16) + k / 32]"),
}


def build_mutant(tmp_path, name):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"{name}: the text to mutate is not unique in oracle.c"
    src = tmp_path / f"oracle_{name}.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / f"liboracle_{name}.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(lib), str(src), "-lm"], check=True)
    return str(lib)


def run_pins(lib_path):
    env = dict(os.environ, ORACLE_LIB=lib_path)
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)


def test_unmutated_copy_passes_the_pins(tmp_path):
    # the harness itself: an untouched copy built the same way passes
    src = tmp_path / "oracle_copy.c"
    src.write_text(open(SRC).read())
    lib = tmp_path / "liboracle_copy.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", str(lib), str(src), "-lm"], check=True)
    r = run_pins(str(lib))
    assert r.returncode == 0, r.stdout[-3000:]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(tmp_path, name):
    r = run_pins(build_mutant(tmp_path, name))
    assert r.returncode == 1, f"{name}: the pins did not catch it\n{r.stdout[-3000:]}"
    assert " failed" in r.stdout, r.stdout[-3000:]
