"""Mutation check of the oracle's pins.

Each case plants one plausible mistake in a private copy of the oracle's C
source (a dropped term, a wrong sign, a transposed operand, a wrong leading
dimension, a wrong widening), compiles it to a temporary library and requires
that at least one pin fails.  The committed oracle is never modified.
"""
import os

import numpy as np

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "gemm_oracle.c")

MUTANTS = {
    "dropped_beta_term": ("value = value + beta * c_old;", "value = value;"),
    "beta_sign": ("value = value + beta * c_old;", "value = value - beta * c_old;"),
    "product_sign": ("acc[j] = acc[j] + a * b;", "acc[j] = acc[j] - a * b;"),
    "b_transposed": ("const double b = (double)b_row[j];",
                     "const double b = (double)B[j * ldb + k];"),
    "a_uses_K_not_lda": ("const float *a_row = A + i * lda;", "const float *a_row = A + i * K;"),
    "alpha_ignored": ("value = alpha * acc[j];", "value = acc[j];"),
    "den_signed": ("mag[j] = mag[j] + abs_a * fabs(b);", "mag[j] = mag[j] + a * b;"),
    "beta_zero_reads_c": ("if (beta != 0.0) {\n            double c_old",
                          "if (1) {\n            double c_old"),
    "bf16_wrong_shift": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "k_off_by_one": ("for (int64_t k = 0; k < K; ++k) {\n                    const double a = (double)",
                     "for (int64_t k = 1; k < K; ++k) {\n                    const double a = (double)"),
}


_CHILD = r"""
import sys
sys.path[:0] = [%r, %r]
import oracle
from oracle_pins import ALL_PINS
orc = oracle.OracleLib(%r)
failed = []
for pin in ALL_PINS:
    try:
        pin(orc)
    except Exception:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
"""


def _run_pins_isolated(lib_path):
    """Run every pin against a mutant in a child process (a mutant may crash)."""
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    code = _CHILD % (root, here, lib_path)
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=300)
    if proc.returncode != 0:
        return ["crashed(rc=%d)" % proc.returncode]
    line = [l for l in proc.stdout.splitlines() if l.startswith("FAILED:")][-1]
    return [x for x in line[len("FAILED:"):].split(",") if x]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert old in text, "mutation anchor missing for %s" % name
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new, 1))
    lib_path = oracle.compile_library(str(src), str(tmp_path / "libmutant.so"))
    failed = _run_pins_isolated(lib_path)
    assert failed, "no pin caught mutant %s" % name


# Plausible mistakes in the output conversion of the fused stage, planted by
# swapping oracle.quantize for a wrong version while the pins run.
def _quantize_through_fp32(v, d_type, d_scale=1.0):
    x = np.asarray(v, dtype=np.float32) * np.float32(d_scale)   # rounds twice
    return _QUANTIZE(x.astype(np.float64), d_type, 1.0)


def _quantize_scale_ignored(v, d_type, d_scale=1.0):
    return _QUANTIZE(v, d_type, 1.0)


def _quantize_ties_away(v, d_type, d_scale=1.0):
    x = np.asarray(v, dtype=np.float64) * float(np.float32(d_scale))
    if d_type == "s8":
        r = np.sign(x) * np.floor(np.abs(x) + 0.5)
        return np.clip(np.where(np.isnan(x), 0.0, r), -128, 127).astype(np.int8)
    return _QUANTIZE(v, d_type, d_scale)


_QUANTIZE = oracle.quantize
QUANTIZE_MUTANTS = {
    "rounded_to_fp32_first": _quantize_through_fp32,
    "scale_ignored": _quantize_scale_ignored,
    "s8_ties_away_from_zero": _quantize_ties_away,
}


@pytest.mark.parametrize("name", sorted(QUANTIZE_MUTANTS))
def test_quantize_mutant_is_caught(monkeypatch, name):
    monkeypatch.setattr(oracle, "quantize", QUANTIZE_MUTANTS[name])
    orc = oracle.default()
    failed = []
    for pin in ALL_PINS:
        if "quantize" not in pin.__name__:
            continue
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "no pin caught quantize mutant %s" % name
