"""Pins of the oracle's general TRSM (every side / triangle / op / diagonal
variant, BLAS meaning) against what the mathematics fixes, without a GPU:
 - a dense library solve of the explicitly formed op(A) on tiny inputs
   (numpy.linalg.solve; an independent code path), with NaN in every entry
   the variant must not read;
 - bitwise agreement with the pinned left-lower oracle on that variant;
 - exact integer closed forms (bidiagonal triangles give suffix sums);
 - alpha = 0 gives zeros without reading A."""
import itertools

import numpy as np
import pytest

import oracle

NP = {"f32": np.float32, "f64": np.float64, "c64": np.complex64, "c128": np.complex128}
TOL = {"f32": 2e-6, "f64": 1e-13, "c64": 2e-6, "c128": 1e-13}
VARIANTS = list(itertools.product("LR", "LU", "NTC", "NU"))


def _rand(rng, dtype, shape):
    x = rng.uniform(-1, 1, shape)
    if dtype in ("c64", "c128"):
        x = x + 1j * rng.uniform(-1, 1, shape)
    return x


def _col(x, dtype):
    """Column-major flat buffer of a 2-D array."""
    return np.ascontiguousarray(np.asarray(x, dtype=NP[dtype]).T).ravel()


def _uncol(buf, rows, cols):
    return buf.reshape(cols, rows).T


def _problem(dtype, side, uplo, diag, m, n, seed):
    rng = np.random.default_rng(seed)
    k = m if side == "L" else n
    A = _rand(rng, dtype, (k, k)) / k
    A[np.diag_indices(k)] = 2 + rng.uniform(0, 1, k)  # well conditioned either way
    B = _rand(rng, dtype, (m, n))
    stored = A.astype(complex if dtype in ("c64", "c128") else float).copy()
    unread = np.triu_indices(k, 1) if uplo == "L" else np.tril_indices(k, -1)
    stored[unread] = np.nan
    if diag == "U":
        stored[np.diag_indices(k)] = np.nan
    return A, B, stored


def _dense_reference(A, B, side, uplo, trans, diag, alpha):
    T = np.tril(A) if uplo == "L" else np.triu(A)
    if diag == "U":
        T = T.copy()
        T[np.diag_indices(T.shape[0])] = 1
    if trans == "T":
        T = T.T
    elif trans == "C":
        T = T.conj().T
    if side == "L":
        return np.linalg.solve(T, alpha * B)
    return np.linalg.solve(T.T, (alpha * B).T).T


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
@pytest.mark.parametrize("side,uplo,trans,diag", VARIANTS)
def test_variant_matches_a_dense_solve(dtype, side, uplo, trans, diag):
    m, n = (5, 3) if side == "L" else (3, 5)
    A, B, stored = _problem(dtype, side, uplo, diag, m, n, seed=VARIANTS.index((side, uplo, trans, diag)))
    alpha = (0.75 - 0.5j) if dtype in ("c64", "c128") else 0.75
    a_buf, b_buf = _col(stored, dtype), _col(B, dtype)
    k = A.shape[0]
    oracle.trsm_general(dtype, side, uplo, trans, diag, m, n, alpha, a_buf, k, b_buf, m)
    got = _uncol(b_buf, m, n).astype(np.complex128)
    if dtype in ("f32", "f64") and trans == "C":
        trans_ref = "T"  # A^H of a real matrix is A^T
    else:
        trans_ref = trans
    ref = _dense_reference(A.astype(np.complex128), B.astype(NP[dtype]).astype(np.complex128),
                           side, uplo, trans_ref, diag, alpha)
    assert np.all(np.isfinite(got)), "read an entry outside the variant's triangle or its unit diagonal"
    err = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err < TOL[dtype], f"{side}{uplo}{trans}{diag} {dtype}: {err:.2e}"


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
def test_left_lower_variant_is_the_pinned_oracle_bitwise(dtype):
    rng = np.random.default_rng(3)
    m, n = 9, 4
    A = _rand(rng, dtype, (m, m)) / m
    A[np.diag_indices(m)] += 1.5
    B = _rand(rng, dtype, (m, n))
    a_buf = _col(A, dtype)
    b1, b2 = _col(B, dtype), _col(B, dtype)
    oracle.trsm_general(dtype, "L", "L", "N", "N", m, n, 1.25, a_buf, m, b1, m)
    oracle.trsm_llnn(dtype, m, n, 1.25, a_buf, m, b2, m)
    assert np.array_equal(b1, b2)


def test_bidiagonal_closed_forms():
    """Left, upper, no transpose: T = I - superdiagonal, so T x = b gives the
    suffix sums x_i = b_i + ... + b_{m-1}; right, lower: X T = B with
    T = I - subdiagonal gives the suffix sums along each row."""
    m, n = 7, 6
    B = np.arange(1, m * n + 1, dtype=np.float64).reshape(m, n) % 5 - 2
    U = np.eye(m) - np.eye(m, k=1)
    b = _col(B, "f64")
    oracle.trsm_general("f64", "L", "U", "N", "N", m, n, 1.0, _col(U, "f64"), m, b, m)
    assert np.array_equal(_uncol(b, m, n), np.cumsum(B[::-1], axis=0)[::-1])
    Lo = np.eye(n) - np.eye(n, k=-1)
    b = _col(B, "f64")
    oracle.trsm_general("f64", "R", "L", "N", "N", m, n, 1.0, _col(Lo, "f64"), n, b, m)
    assert np.array_equal(_uncol(b, m, n), np.cumsum(B[:, ::-1], axis=1)[:, ::-1])


def test_zero_alpha_reads_nothing_of_a():
    B = np.ones((4, 3))
    b = _col(B, "f64")
    oracle.trsm_general("f64", "R", "U", "C", "U", 4, 3, 0.0, None, 3, b, 4)
    assert np.array_equal(b, np.zeros(12))
