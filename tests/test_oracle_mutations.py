"""The oracle's pins catch plausible mistakes: each case plants one mistake
in a copy of oracle.c (a dropped term, a wrong operand, a wrong index or
rounding), builds it with the oracle's own flags, runs the pin tests that
should notice against it in a child process, and requires them to fail.
A control run of the unmodified copy must pass.  CPU only; nothing here
touches the product library."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, original text, replacement, pin tests expected to catch it)
MUTATIONS = [
    # RMSNorm + MXCast takes its statistic from x (Eq. (1); MXNorm card Fig. 1
    # caption, left graph): computing it from w = x * gamma instead
    ("rmsnorm statistic of x*gamma",
     "double xj = oracle_bf16_to_double(x[j]);\n            S += xj * xj;\n        }\n"
     "        double r = 1.0 / sqrt(S / (double)D + eps);",
     "double xj = oracle_bf16_to_double(x[j]) * (gamma ? (double)gamma[j] : 1.0);\n"
     "            S += xj * xj;\n        }\n"
     "        double r = 1.0 / sqrt(S / (double)D + eps);",
     ["tests/test_oracle_mx.py::test_rmsnorm_factor_does_not_depend_on_the_gain"]),
    # MXNorm estimates the RMS from the block absmaxes of the cast tensor
    # w = x * gamma (MXNorm card Fig. 1 caption, right graph): using x
    ("mxnorm absmax of x",
     "double v = fabs((double)work[k * B + b]);",
     "double v = fabs(oracle_bf16_to_double(X[t * D + k * B + b]));",
     ["tests/test_oracle_mx.py::test_mxnorm_statistic_is_of_the_cast_tensor",
      "tests/test_oracle_mx.py::test_constant_rows_with_constant_gain"]),
    # S/H uses the full row width (SwiftQK Eq. (1), H_total), not the shard's
    ("qk mean over the shard width",
     "double r = 1.0 / sqrt(S / (double)H + eps);\n        if (rinv) rinv[t] = r;\n"
     "        for (int64_t j = 0; j < H; ++j) {                   /* Phases B, C */\n"
     "            double w = oracle_bf16_to_double(x[j]) * (double)gamma[j];",
     "double r = 1.0 / sqrt(S / (double)W + eps);\n        if (rinv) rinv[t] = r;\n"
     "        for (int64_t j = 0; j < H; ++j) {                   /* Phases B, C */\n"
     "            double w = oracle_bf16_to_double(x[j]) * (double)gamma[j];",
     ["tests/test_oracle_qk.py::test_worked_example_eqs_2_to_8",
      "tests/test_oracle_qk.py::test_split_equals_unsplit"]),
    # eps inside the square root, added to the mean square (Eq. (1))
    ("qk eps outside the root",
     "double r = 1.0 / sqrt(S / (double)H + eps);\n        if (rinv) rinv[t] = r;\n"
     "        for (int64_t j = 0; j < H; ++j) {                   /* Phases B, C */\n"
     "            double w = oracle_bf16_to_double(x[j]) * (double)gamma[j];",
     "double r = 1.0 / (sqrt(S / (double)H) + eps);\n        if (rinv) rinv[t] = r;\n"
     "        for (int64_t j = 0; j < H; ++j) {                   /* Phases B, C */\n"
     "            double w = oracle_bf16_to_double(x[j]) * (double)gamma[j];",
     ["tests/test_oracle_qk.py::test_constant_row_closed_form"]),
    # the gain multiplies each element (Algorithm 1): a shifted gain index
    ("qk gain of the wrong channel",
     "/* Phases B, C */\n            double w = oracle_bf16_to_double(x[j]) * (double)gamma[j];",
     "/* Phases B, C */\n            double w = oracle_bf16_to_double(x[j]) * (double)gamma[(j + 1) % H];",
     ["tests/test_oracle_qk.py::test_constant_row_closed_form"]),
    # E8M0 scale: round(log2 .), not floor (MXNorm card Fig. 1 caption)
    ("e8m0 floor instead of round",
     "return E + (fma(m, m, -2.0) > 0.0 ? 1 : 0);",
     "return E;",
     ["tests/test_oracle_formats.py::test_round_log2_against_double_log2_on_every_fp32_exponent",
      "tests/test_oracle_mx.py::test_block_stage_brute_force"]),
    # MXNorm p = 2: the root of the mean of squared absmaxes, then c(B, 2)
    ("mxnorm p=2 without the root",
     "double Mp = p == 1 ? acc / (double)K : sqrt(acc / (double)K);",
     "double Mp = acc / (double)K;",
     ["tests/test_oracle_mx.py::test_gaussian_invariance",
      "tests/test_oracle_mx.py::test_constant_rows_closed_form"]),
]


def build_variant(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    return oracle.compile_source(str(src), str(tmp_path / f"{name}.so"))


def run_pins(lib, pins):
    env = dict(os.environ, NTS_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "not gpu",
                        "-p", "no:cacheprovider", *pins],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def test_unmodified_copy_passes_the_pins(tmp_path):
    pins = sorted({p for m in MUTATIONS for p in m[3]})
    lib = build_variant(tmp_path, "control", open(SRC).read())
    rc, out = run_pins(lib, pins)
    assert rc == 0, out


@pytest.mark.parametrize("name,old,new,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, pins):
    text = open(SRC).read()
    assert text.count(old) == 1, f"the oracle no longer contains the text of '{name}'"
    lib = build_variant(tmp_path, "mutant", text.replace(old, new))
    rc, out = run_pins(lib, pins)
    assert rc != 0, f"no pin noticed '{name}':\n{out}"
