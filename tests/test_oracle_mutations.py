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
