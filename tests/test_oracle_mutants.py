"""Strength of the oracle pins: each planted mistake must fail a pin.

A copy of the oracle source with one plausible mistake is compiled into a
temporary library, and the pins run against it in a child process (a planted
index error may read out of bounds; the child absorbs that).  A mutant that
passes every pin would mean the pins cannot tell that mistake from the
definition.
"""

import os
import subprocess
import sys
import textwrap

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in sgemm_oracle.c, replacement)
MUTANTS = [
    ("dropped_last_k", "for (int64_t k = 0; k < K; ++k) {",
     "for (int64_t k = 0; k < K - 1; ++k) {"),
    ("beta_sign", "v += (double)beta * (double)C0[i * ldc + j];",
     "v -= (double)beta * (double)C0[i * ldc + j];"),
    ("transposed_A", "const double a = (double)A[i * lda + k];",
     "const double a = (double)A[(k % M) * lda + (i % K)];"),
    ("wrong_ld_for_B", "const float *brow = B + k * ldb;",
     "const float *brow = B + k * N;"),
    ("fp32_accumulate", "acc[j] += a * (double)brow[j];",
     "acc[j] = (float)((float)acc[j] + (float)a * brow[j]);"),
    ("alpha_dropped", "double v = use_ab ? (double)alpha * acc[j] : 0.0;",
     "double v = use_ab ? acc[j] : 0.0;"),
    ("beta_zero_reads_C0", "const int use_c = (beta != 0.0f);",
     "const int use_c = (C0 != NULL);"),
    ("row_off_by_one", "const int64_t i = rows[r];",
     "const int64_t i = (rows[r] + 1) % M;"),
    ("alpha_zero_reads_AB", "const int use_ab = (alpha != 0.0f) && (K > 0);",
     "const int use_ab = (K > 0);"),
    ("column_shift", "acc[j] += a * (double)brow[j];",
     "acc[j] += a * (double)brow[(j + 1) % N];"),
    ("tf32_truncates", "u = (u + 0x1000u) & 0xffffe000u;", "u = u & 0xffffe000u;"),
    ("tf32_ties_even", "u = (u + 0x1000u) & 0xffffe000u;",
     "u = (u + 0x0fffu + ((u >> 13) & 1u)) & 0xffffe000u;"),
    ("tf32_keeps_11_bits", "u = (u + 0x1000u) & 0xffffe000u;", "u = (u + 0x0800u) & 0xfffff000u;"),
    ("bf16_ties_away", "u = (u + 0x7fffu + ((u >> 16) & 1u)) & 0xffff0000u;",
     "u = (u + 0x8000u) & 0xffff0000u;"),
    ("bf16_truncates", "u = (u + 0x7fffu + ((u >> 16) & 1u)) & 0xffff0000u;", "u = u & 0xffff0000u;"),
    ("bias_by_row", "v += (double)bias[j];", "v += (double)bias[i % N];"),
    ("act_before_bias", "orow[j] = (float)activate(v, act);",
     "orow[j] = (float)(activate(v - (bias ? (double)bias[j] : 0.0), act) + (bias ? (double)bias[j] : 0.0));"),
    ("gelu_coefficient", "(x + 0.044715 * x * x * x)", "(x + 0.04715 * x * x * x)"),
    ("silu_sign", "return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    ("relu_nan_to_zero", "return x < 0.0 ? 0.0 : x;", "return x > 0.0 ? x : 0.0;"),
]

CHILD = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle, pins
    orc = oracle.Oracle({lib!r})
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError as e:
            failed.append(pin.__name__)
    print("FAILED_PINS", ",".join(failed))
    sys.exit(0 if failed else 1)
""")


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut = tmp_path / f"{name}.c"
    mut.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mut), str(tmp_path / f"lib{name}.so"))
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300, env={**os.environ, "OMP_NUM_THREADS": "2"})
    # Exit 0 with a list of failing pins, or a crash: either way the mutant
    # did not pass.  Exit 1 means every pin passed -- the mistake went unseen.
    assert r.returncode != 1, f"mutant {name} passed every pin:\n{r.stdout}\n{r.stderr}"
