"""The pins must fail on a wrong oracle.  Each case plants one plausible
mistake (a flipped sign, a transposed or shifted index, a dropped term or
factor, a wrong complex formula, a wrong layout) in a temporary copy of the
oracle source, rebuilds it in a scratch folder and runs the pin suite against
it in a subprocess: every mutant must make at least one pin fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "trsm_oracle.c")

MUTANTS = [
    ("si[c] -= l * xk[c]", "si[c] += l * xk[c]"),
    ("const double l = ld_real(A, dtype, off(layout, lda, i, k));",
     "const double l = ld_real(A, dtype, off(layout, lda, k, i));"),
    ("xk[c] = xk[c] / d;", "xk[c] = xk[c] * d;"),
    ("for (int64_t i = k + 1; i < m; ++i) {\n            const double l",
     "for (int64_t i = k + 2; i < m; ++i) {\n            const double l"),
    ("r.im = a.re * b.im + a.im * b.re;", "r.im = a.re * b.im - a.im * b.re;"),
    ("s[i * w + c] = alpha * ld_real", "s[i * w + c] = ld_real"),
    ("r.im = (a.im - a.re * q) / den;", "r.im = (a.im + a.re * q) / den;"),
    ("r.re = (a.re * q + a.im) / den;", "r.re = (a.re * q - a.im) / den;"),
    ("const ocplx l = ld_cplx(A, dtype, off(layout, lda, i, k));",
     "const ocplx l = ld_cplx(A, dtype, off(layout, lda, i, k + 1));"),
    ("const ocplx d = ld_cplx(A, dtype, off(layout, lda, k, k));",
     "const ocplx d = ld_cplx(A, dtype, off(layout, lda, k, k > 0 ? k - 1 : 0));"),
    ("return layout == OR_COL_MAJOR ? col * ld + row : row * ld + col;",
     "return layout == OR_COL_MAJOR ? col * ld + row : col * ld + row;"),
]


# mistakes in the general-variant solve, caught by tests/test_oracle_variants.py
VARIANT_MUTANTS = [
    ("if (trans == 2) v.im = -v.im;", "if (trans == 1) v.im = -v.im;"),          # conjugates the wrong op
    ("const int64_t r = trans ? j : i, c = trans ? i : j;",
     "const int64_t r = i, c = j;"),                                               # transpose dropped
    ("const int lower_system = side == 0 ? t_lower : !t_lower;",
     "const int lower_system = t_lower;"),                                          # right side solved as left
    ("if (i == j && diag == 1) {", "if (i == j && diag == 2) {"),                 # unit diagonal ignored
    ("acc = c_sub(acc, c_mul(tv, x[q]));", "acc = c_sub(acc, c_mul(tv, x[j]));"),  # wrong index
]


def _run_pins_on_mutant(tmp_path, before, after, pin_file):
    src = open(SRC).read()
    assert before in src, "mutation anchor no longer in the oracle source"
    mutant = tmp_path / "trsm_oracle.c"
    mutant.write_text(src.replace(before, after, 1))
    env = dict(os.environ, TRSM_ORACLE_TEST_SRC=str(mutant),
               TRSM_ORACLE_TEST_BUILD=str(tmp_path / "build"))
    return subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", pin_file)],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


@pytest.mark.parametrize("idx", range(len(VARIANT_MUTANTS)))
def test_variant_pins_reject_planted_mistake(tmp_path, idx):
    r = _run_pins_on_mutant(tmp_path, *VARIANT_MUTANTS[idx], "test_oracle_variants.py")
    assert r.returncode == 1 and "failed" in r.stdout, r.stdout[-2000:]


@pytest.mark.parametrize("idx", range(len(MUTANTS)))
def test_pins_reject_planted_mistake(tmp_path, idx):
    before, after = MUTANTS[idx]
    src = open(SRC).read()
    assert before in src, "mutation anchor no longer in the oracle source"
    mutant = tmp_path / "trsm_oracle.c"
    mutant.write_text(src.replace(before, after, 1))
    env = dict(os.environ, TRSM_ORACLE_TEST_SRC=str(mutant),
               TRSM_ORACLE_TEST_BUILD=str(tmp_path / "build"))
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle_pins.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1 and "failed" in r.stdout, r.stdout[-2000:]
