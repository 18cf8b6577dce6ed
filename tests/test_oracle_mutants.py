"""Planted mistakes in the oracle must fail its pins (no GPU).

Each case copies oracle_gemm.c, plants one plausible mistake (a dropped term,
a wrong sign, a transposed index, a wrong constant, a misplaced epilogue
step), compiles it with gcc into a temporary library, and runs the pin suite
against it in a subprocess.  The suite must fail for every mutant; the
unmodified source must pass (covered by test_oracle_pins itself).
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle_gemm.c")

MUTANTS = {
    "drop_first_k_term": ("for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 1; k < K; ++k) {"),
    "wrong_beta_sign": ("v += beta * mat(", "v -= beta * mat("),
    "transposed_index": ("*rs = layout == OR_ROW ? ld : 1;", "*rs = layout == OR_ROW ? 1 : ld;"),
    "batch_stride_ignored": ("int64_t idx = b * stride + ", "int64_t idx = 0 * stride + "),
    "alpha_dropped": ("double v = alpha * acc;", "double v = acc;"),
    "beta_zero_reads_C": ("if (beta != 0.0) v += beta", "v += beta"),
    "gelu_cubic_constant": ("0.044715 * x * x * x", "0.04715 * x * x * x"),
    "gelu_scale_constant": ("sqrt(2.0 / M_PI)", "sqrt(1.0 / M_PI)"),
    "bias_after_activation": (
        "    if (bias) v += (double)bias[bias_rows ? i : j];\n    if (act == OR_ACT_GELU_TANH) v = oracle_gelu_tanh(v);",
        "    if (act == OR_ACT_GELU_TANH) v = oracle_gelu_tanh(v);\n    if (bias) v += (double)bias[bias_rows ? i : j];"),
    "bf16_shift": ("(uint32_t)h << 16", "(uint32_t)h << 15"),
    "f16_exponent_bias": ("e - 25", "e - 24"),
    "f16_subnormal_scale": ("ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    "k_loop_reversed_operands": ("mat(B, ab_dt, brs, bcs, sb, b, k, j);", "mat(B, ab_dt, brs, bcs, sb, b, j, k);"),
    "relu_passes_negatives": ("return x > 0.0 ? x : 0.0;", "return x > 0.0 ? x : -x;"),
    "gelu_erf_scale": ("erf(x / sqrt(2.0))", "erf(x / 2.0)"),
    "bias_orientation_swapped": ("bias[bias_rows ? i : j]", "bias[bias_rows ? j : i]"),
    "sampled_last_k_dropped": ("for (int64_t k = 0; k < K; ++k)\n            acc +=",
                               "for (int64_t k = 0; k + 1 < K; ++k)\n            acc +="),
    "strided_column_stride_dropped": ("int64_t idx = b * stride + r * rs + c * cs;", "int64_t idx = b * stride + r * rs + c;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    # the site must be code, not the header comment
    assert src.index(old) > src.index("#include"), f"mutation site for {name} is in a comment"
    mutated = src.replace(old, new, 1)
    csrc = tmp_path / "oracle_mut.c"
    csrc.write_text(mutated)
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared", "-o",
                    str(lib), str(csrc), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
