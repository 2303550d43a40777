"""The oracle's pins catch plausible mistakes.

Each case copies the oracle's C source, plants one mistake of the kind a
careful reader could still make (a dropped sign, a wrong exponent bias, a
round-half-up tie, a reciprocal multiply in place of the division, a wrong
scale index, a transposed operand, a dropped block, a double rounding), builds
it with gcc and runs the pin tests against it in a fresh process. Every
mutant must make at least one pin fail. The planted mistakes live only in a
temporary copy on the CPU.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "fp8_block_oracle.c")

MUTANTS = {
    "decode_drops_sign": ("        if (s) v = -v;\n", "\n"),
    "decode_subnormal_exponent": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "decode_bias_8": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "encode_ties_up": ("else code = (lo & 1) ? hi : lo;", "else code = hi;"),
    "encode_no_saturation": ("return sign | 0x7E; /* satfinite */", "return sign | 0x7F; /* satfinite */"),
    "quant_reciprocal_multiply": ("float t = v / s;", "float t = v * (1.0f / s);"),
    "quant_scale_max_440": ("amax / E4M3_MAX;", "amax / 440.0f;"),
    "gemm_sw_index_swapped": ("sw[(n / G) * KB + kb]", "sw[kb * ((N + G - 1) / G) + n / G]"),
    "gemm_sa_ignores_row": ("(double)sa[m * KB + kb]", "(double)sa[kb]"),
    "gemm_w_transposed": ("P += (int64_t)e4m3_int[qr[k]] * (int64_t)e4m3_int[wr[k]];",
                          "P += (int64_t)e4m3_int[qr[k]] * (int64_t)e4m3_int[w[k * N + n]];"),
    "gemm_drops_first_block": ("for (int64_t kb = 0; kb < KB; ++kb) {\n                int64_t P = 0;",
                               "for (int64_t kb = 1; kb < KB; ++kb) {\n                int64_t P = 0;"),
    "gemm_abs_sign": ("acc += term;", "acc += fabs(term);"),
    "bf16_double_rounding": ("frexp(y, &e);", "y = (double)(float)y; frexp(y, &e);"),
    "bf16_truncates": ("nearbyint(ldexp(y, -qe))", "trunc(ldexp(y, -qe))"),
    "w8a16_sw_ignores_row_block": ("sw_row = sw + (n / G) * KB;", "sw_row = sw;"),
    "w8a16_drops_activation_sign": ("dot += (double)bf16_to_float(xr[k])", "dot += fabs((double)bf16_to_float(xr[k]))"),
    "w8a16_drops_last_block_element": ("for (int64_t k = kb * G; k < (kb + 1) * G; ++k)\n                    dot",
                                       "for (int64_t k = kb * G; k < (kb + 1) * G - 1; ++k)\n                    dot"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new), encoding="utf-8")
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
                    "-ffp-contract=off", str(mutant), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, FP8_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout or "error" in r.stdout.lower()
