"""The oracle's pins are strong enough to catch plausible mistakes.

Each mutant is a copy of oracle.c with one planted mistake (a transposed
operand, a dropped term, a wrong sign or index, a missing absolute value, a
leading dimension ignored, a narrower accumulator). It is compiled on the CPU
and the full pin suite of test_oracle.py runs against it in a child process
(a mutant may read out of bounds, which must not take the test run down).
Every mutant must fail at least one pin; the unmodified copy must pass all.
"""

import os
import subprocess
import sys
import tempfile

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "none": [],
    "gemm_transposed_A": [("j->A[i * j->lda + k]", "j->A[k * j->lda + i]")],
    "gemm_drops_last_term": [("for (int64_t k = 0; k < j->K; ++k) {",
                              "for (int64_t k = 0; k + 1 < j->K; ++k) {")],
    "gemm_drops_first_term": [("for (int64_t k = 0; k < j->K; ++k) {",
                               "for (int64_t k = 1; k < j->K; ++k) {")],
    "gemm_wrong_sign": [("c[col] += p;", "c[col] -= p;")],
    "gemm_wrong_B_column": [("const double p = a * b[col];",
                             "const double p = a * b[(col + 1) % j->N];")],
    "gemm_E_without_abs": [("if (e) e[col] += fabs(p);", "if (e) e[col] += p;")],
    "gemm_ldc_ignored": [("double *c = j->C + i * j->ldc;", "double *c = j->C + i * j->N;")],
    "gemm_lda_ignored": [("j->A[i * j->lda + k]", "j->A[i * j->K + k]")],
    "gemv_transposed_A": [("A[i * lda + j] * x[j]", "A[j * lda + i] * x[j]")],
    "gemv_drops_first_term": [("for (int64_t j = 0; j < N; ++j) {",
                               "for (int64_t j = 1; j < N; ++j) {")],
    "gemv_wrong_x_index": [("A[i * lda + j] * x[j]", "A[i * lda + j] * x[i % N]")],
    "gemv_float_accumulator": [("double sum = 0.0, mag = 0.0;",
                                "float sum = 0.0f; double mag = 0.0;")],
    "bias_on_wrong_axis": [("if (bias) v += bias_per_column ? bias[j] : bias[i];",
                            "if (bias) v += bias_per_column ? bias[i % N] : bias[j % M];")],
    "bias_subtracted": [("if (bias) v += bias_per_column ? bias[j] : bias[i];",
                         "if (bias) v -= bias_per_column ? bias[j] : bias[i];")],
    "relu_as_abs": [("if (act == 1 && v < 0.0) v = 0.0;", "if (act == 1 && v < 0.0) v = -v;")],
    "conv_kernel_axes_swapped": [("const double *w = j->Wt + (kh * j->KW + kw) * j->C * j->CO + co;",
                                  "const double *w = j->Wt + (kw * j->KH + kh) * j->C * j->CO + co;")],
    "conv_padding_ignored": [("const int64_t ih = oh * j->sh - j->ph + kh * j->dh;",
                              "const int64_t ih = oh * j->sh + kh * j->dh;")],
    "conv_column_stride_ignored": [("const int64_t iw = ow * j->sw - j->pw + kw * j->dw;",
                                    "const int64_t iw = ow - j->pw + kw * j->dw;")],
    "conv_row_dilation_ignored": [("const int64_t ih = oh * j->sh - j->ph + kh * j->dh;",
                                   "const int64_t ih = oh * j->sh - j->ph + kh;")],
    "conv_weights_as_co_ci": [("const double *w = j->Wt + (kh * j->KW + kw) * j->C * j->CO + co;",
                               "const double *w = j->Wt + (kh * j->KW + kw) * j->C * j->CO + co * j->C;"),
                              ("const double p = x[ci] * w[ci * j->CO];", "const double p = x[ci] * w[ci];")],
    "conv_column_bound_off_by_one": [("if (iw < 0 || iw >= j->W) continue;", "if (iw < 0 || iw > j->W) continue;")],
    "conv_E_without_abs": [("sum += p;\n                            mag += fabs(p);",
                            "sum += p;\n                            mag += p;")],
    "relu_before_bias": [("            double v = C[i * ldc + j];\n            if (bias) v += bias_per_column ? bias[j] : bias[i];\n            if (act == 1 && v < 0.0) v = 0.0;",
                          "            double v = C[i * ldc + j];\n            if (act == 1 && v < 0.0) v = 0.0;\n            if (bias) v += bias_per_column ? bias[j] : bias[i];")],
}

RUNNER = r"""
import sys
sys.path.insert(0, {root!r})
import oracle
from tests import test_oracle as t
lib = oracle.load({lib!r})
failed = []
for pin in t.PINS:
    try:
        pin(lib)
    except Exception as e:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
sys.exit(1 if failed else 0)
"""


def _build_mutant(tmp, name, edits):
    with open(SRC) as f:
        src = f.read()
    for old, new in edits:
        assert old in src, f"mutation anchor missing for {name}: {old!r}"
        src = src.replace(old, new)
    c_path = os.path.join(tmp, f"{name}.c")
    with open(c_path, "w") as f:
        f.write(src)
    h = os.path.join(ROOT, "oracle", "oracle.h")
    with open(h) as f, open(os.path.join(tmp, "oracle.h"), "w") as g:
        g.write(f.read())
    return oracle.build(src=c_path, out=os.path.join(tmp, f"lib{name}.so"))


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    lib = _build_mutant(str(tmp_path), name, MUTANTS[name])
    proc = subprocess.run([sys.executable, "-c", RUNNER.format(root=ROOT, lib=lib)],
                          capture_output=True, text=True, timeout=300, cwd=ROOT)
    if name == "none":
        assert proc.returncode == 0, proc.stdout + proc.stderr
    else:
        # a non-zero exit (a failed pin, or a crash) means the mistake was caught
        assert proc.returncode != 0, f"planted mistake {name} passed every pin"
