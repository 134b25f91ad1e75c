"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself (special cases, exact integer arithmetic, closed forms, an
independent brute-force elimination, LAPACK, and the backward-error bound).

The solve being pinned is X = L^{-1}(alpha B) with L lower triangular,
non-unit diagonal ("Hierarchical Shared Memory-Aware Optimization for TRSM on
GPU Platforms": left-side lower-triangular TRSM; llama.cpp PR 17457 "SOLVE_TRI
CUDA kernel for small matrices": forward substitution, no zero-pivot guard).
"""
import numpy as np
import pytest

import trsm_inputs as ti
from oracle_util import oracle_solve, rel_fro, residual

DTYPES = ["f32", "f64", "c64", "c128"]
EPS = {"f32": 2.0 ** -24, "f64": 2.0 ** -53, "c64": 2.0 ** -24, "c128": 2.0 ** -53}


def _rng(seed=1234):
    return np.random.default_rng(seed)


def _rand(rng, shape, dtype, lo=-1.0, hi=1.0):
    x = rng.uniform(lo, hi, shape)
    if ti.IS_COMPLEX[dtype]:
        x = x + 1j * rng.uniform(lo, hi, shape)
    return x.astype(ti.NUMPY[dtype])


def _alpha_times(alpha, B, dtype):
    """alpha * B with one rounding per real operation (no fused multiply-add)."""
    if ti.IS_COMPLEX[dtype]:
        a = complex(alpha)
        br = B.real.astype(np.float64)
        bi = B.imag.astype(np.float64)
        re = np.multiply(a.real, br) - np.multiply(a.imag, bi)
        im = np.multiply(a.real, bi) + np.multiply(a.imag, br)
        return (re + 1j * im).astype(ti.NUMPY[dtype])
    return (np.float64(alpha) * B.astype(np.float64)).astype(ti.NUMPY[dtype])


# ---------------------------------------------------------------- special cases
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("layout", ["col", "row"])
def test_identity_gives_alpha_b(oracle_mod, dtype, layout):
    rng = _rng()
    m, n, batch = 37, 5, 3
    L = np.broadcast_to(np.eye(m), (batch, m, m)).astype(ti.NUMPY[dtype])
    B = _rand(rng, (batch, m, n), dtype)
    alpha = (0.75 - 1.25j) if ti.IS_COMPLEX[dtype] else 1.5
    X, _, _ = oracle_solve(oracle_mod, dtype, L, B, alpha, layout=layout)
    np.testing.assert_array_equal(X, _alpha_times(alpha, B, dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_diagonal_divides(oracle_mod, dtype):
    rng = _rng(7)
    m, n, batch = 23, 4, 2
    d = _rand(rng, (batch, m), dtype, 0.5, 2.0)
    L = np.zeros((batch, m, m), dtype=ti.NUMPY[dtype])
    idx = np.arange(m)
    L[:, idx, idx] = d
    B = _rand(rng, (batch, m, n), dtype)
    alpha = (2.0 + 0.5j) if ti.IS_COMPLEX[dtype] else -0.5
    X, _, _ = oracle_solve(oracle_mod, dtype, L, B, alpha)
    t = np.complex128 if ti.IS_COMPLEX[dtype] else np.float64
    ref = (t(alpha) * B.astype(t)) / d.astype(t)[:, :, None]
    err = np.abs(X.astype(t) - ref) / np.abs(ref)
    assert err.max() <= 4 * EPS[dtype]


def test_alpha_zero_does_not_read_a(oracle_mod):
    m, n = 9, 3
    for dtype in DTYPES:
        A = np.full(m * m, np.nan, dtype=ti.NUMPY[dtype])
        B = np.full(m * n, 3.0, dtype=ti.NUMPY[dtype])
        oracle_mod.trsm_llnn(dtype, m, n, 0.0, A, m, B, m)
        assert np.all(B == 0)
        oracle_mod.trsm_llnn(dtype, m, n, 0.0, None, m, B, m)


def test_quick_returns_leave_b_untouched(oracle_mod):
    B = np.arange(12, dtype=np.float64)
    A = np.full(16, np.nan)
    before = B.copy()
    oracle_mod.trsm_llnn("f64", 0, 3, 1.0, A, 1, B, 1)
    oracle_mod.trsm_llnn("f64", 4, 0, 1.0, A, 4, B, 4)
    oracle_mod.trsm_llnn("f64", 3, 4, 1.0, A, 3, B, 3, batch=0)
    np.testing.assert_array_equal(B, before)


@pytest.mark.parametrize("dtype", DTYPES)
def test_m_equals_one(oracle_mod, dtype):
    rng = _rng(3)
    L = _rand(rng, (4, 1, 1), dtype, 1.0, 2.0)
    B = _rand(rng, (4, 1, 6), dtype)
    X, _, _ = oracle_solve(oracle_mod, dtype, L, B, 1.0)
    t = np.complex128 if ti.IS_COMPLEX[dtype] else np.float64
    ref = B.astype(t) / L.astype(t)
    assert np.abs(X.astype(t) - ref).max() <= 4 * EPS[dtype] * np.abs(ref).max()


def test_zero_diagonal_propagates_ieee(oracle_mod):
    m, n = 4, 2
    L = np.tril(np.ones((1, m, m)))
    L[0, 1, 1] = 0.0
    B = np.ones((1, m, n))
    X, _, _ = oracle_solve(oracle_mod, "f64", L, B, 1.0)
    assert np.all(np.isfinite(X[0, 0]))
    assert not np.any(np.isfinite(X[0, 1:]))


# ---------------------------------------------------------------- exact integers
def _integer_system(rng, dtype, batch, m, n):
    """Lower L with entries in {-1,0,1} and a power-of-two (or unit Gaussian)
    diagonal, integer X with |x| <= 8, and B = L X computed exactly in int64."""
    cplx = ti.IS_COMPLEX[dtype]
    lre = rng.integers(-1, 2, (batch, m, m))
    xre = rng.integers(-8, 9, (batch, m, n))
    if cplx:
        lim = rng.integers(-1, 2, (batch, m, m))
        xim = rng.integers(-8, 9, (batch, m, n))
        diag = np.array([1, -1, 1j, -1j, 2, -2j, 1 + 1j])
    else:
        lim = np.zeros_like(lre)
        xim = np.zeros_like(xre)
        diag = np.array([1, -1, 2, -2, 4])
    tri = np.tril(np.ones((m, m), dtype=np.int64), -1)
    lre *= tri
    lim *= tri
    dsel = diag[rng.integers(0, diag.size, (batch, m))]
    idx = np.arange(m)
    lre[:, idx, idx] = dsel.real.astype(np.int64)
    lim[:, idx, idx] = dsel.imag.astype(np.int64)
    bre = lre @ xre - lim @ xim
    bim = lre @ xim + lim @ xre
    t = ti.NUMPY[dtype]
    if cplx:
        L = (lre + 1j * lim).astype(t)
        X = (xre + 1j * xim).astype(t)
        B = (bre + 1j * bim).astype(t)
    else:
        L, X, B = lre.astype(t), xre.astype(t), bre.astype(t)
    return L, X, B


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("layout", ["col", "row"])
@pytest.mark.parametrize("m,n", [(1, 1), (2, 3), (7, 17), (64, 6), (130, 5)])
def test_integer_exact_recovery(oracle_mod, dtype, layout, m, n):
    rng = _rng(m * 31 + n)
    batch = 3
    L, X, B = _integer_system(rng, dtype, batch, m, n)
    lda = m + 3
    ldb = (m if layout == "col" else n) + 2
    major_b = n if layout == "col" else m
    sa = m * lda + 5
    sb = major_b * ldb + 7
    Xo, raw, geo = oracle_solve(oracle_mod, dtype, L, B, 1.0, layout=layout, lda=lda,
                                ldb=ldb, stride_a=sa, stride_b=sb)
    np.testing.assert_array_equal(Xo, X)
    # padding of B (beyond ld and between systems) is never written
    mask = np.isnan(ti.to_storage(np.zeros_like(B), layout, ldb, sb))
    assert np.all(np.isnan(raw[mask]))


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("dtype", DTYPES)
def test_bidiagonal_gives_prefix_sum(oracle_mod, dtype):
    """L = I - (sub-diagonal of ones): x_i = x_{i-1} + alpha b_i, i.e. alpha
    times the running sum of B down each column."""
    rng = _rng(11)
    m, n, batch = 300, 4, 2
    L = np.zeros((batch, m, m), dtype=ti.NUMPY[dtype])
    idx = np.arange(m)
    L[:, idx, idx] = 1
    L[:, idx[1:], idx[:-1]] = -1
    Bi = rng.integers(-8, 9, (batch, m, n)).astype(np.float64)
    if ti.IS_COMPLEX[dtype]:
        Bi = Bi + 1j * rng.integers(-8, 9, (batch, m, n))
    B = Bi.astype(ti.NUMPY[dtype])
    X, _, _ = oracle_solve(oracle_mod, dtype, L, B, 1.5)
    np.testing.assert_array_equal(X, (1.5 * np.cumsum(Bi, axis=1)).astype(B.dtype))


@pytest.mark.parametrize("dtype", DTYPES)
def test_all_ones_lower_gives_first_difference(oracle_mod, dtype):
    """L = all-ones lower triangle: sum_{k<=i} x_k = alpha b_i, so
    x_0 = alpha b_0 and x_i = alpha (b_i - b_{i-1})."""
    rng = _rng(12)
    m, n, batch = 257, 3, 2
    L = np.broadcast_to(np.tril(np.ones((m, m))), (batch, m, m)).astype(ti.NUMPY[dtype])
    Bi = rng.integers(-8, 9, (batch, m, n)).astype(np.float64)
    if ti.IS_COMPLEX[dtype]:
        Bi = Bi + 1j * rng.integers(-8, 9, (batch, m, n))
    B = Bi.astype(ti.NUMPY[dtype])
    X, _, _ = oracle_solve(oracle_mod, dtype, L, B, -2.0)
    ref = -2.0 * np.diff(Bi, axis=1, prepend=0)
    np.testing.assert_array_equal(X, ref.astype(B.dtype))


# ---------------------------------------------------------------- brute force
def _ge_partial_pivot(A, B):
    """Gaussian elimination with partial pivoting on the full square matrix
    (rows swapped by the largest modulus in each column), then back
    substitution.  Pure Python; an independent route to A^{-1} B."""
    m = len(A)
    n = len(B[0])
    M = [list(A[i]) + list(B[i]) for i in range(m)]
    for c in range(m):
        p = max(range(c, m), key=lambda r: abs(M[r][c]))
        M[c], M[p] = M[p], M[c]
        for r in range(c + 1, m):
            f = M[r][c] / M[c][c]
            for q in range(c, m + n):
                M[r][q] = M[r][q] - f * M[c][q]
    X = [[0.0] * n for _ in range(m)]
    for j in range(n):
        for i in range(m - 1, -1, -1):
            s = M[i][m + j]
            for k in range(i + 1, m):
                s = s - M[i][k] * X[k][j]
            X[i][j] = s / M[i][i]
    return X


@pytest.mark.parametrize("dtype", ["f64", "c128"])
@pytest.mark.parametrize("m", [1, 2, 3, 5, 8])
def test_brute_force_elimination_small(oracle_mod, dtype, m):
    rng = _rng(100 + m)
    n, batch = 3, 4
    # large off-diagonal entries so that partial pivoting really swaps rows
    L = _rand(rng, (batch, m, m), dtype, -3.0, 3.0)
    L = np.tril(L)
    idx = np.arange(m)
    L[:, idx, idx] = _rand(rng, (batch, m), dtype, 0.5, 1.5)
    B = _rand(rng, (batch, m, n), dtype)
    alpha = (1.25 + 0.5j) if ti.IS_COMPLEX[dtype] else 1.25
    X, _, _ = oracle_solve(oracle_mod, dtype, L, B, alpha)
    for b in range(batch):
        ref = np.array(_ge_partial_pivot(L[b].tolist(), (alpha * B[b]).tolist()))
        assert rel_fro(X[b], ref) <= 1e-12


@pytest.mark.parametrize("dtype", DTYPES)
def test_matches_lapack_triangular_solve(oracle_mod, dtype):
    sl = pytest.importorskip("scipy.linalg")
    L, B = ti.generate(dtype, 200, 33, batch=2, kind="dd64", seed=5)
    alpha = (0.5 + 1j) if ti.IS_COMPLEX[dtype] else 0.5
    X, _, _ = oracle_solve(oracle_mod, dtype, L, B, alpha)
    t = np.complex128 if ti.IS_COMPLEX[dtype] else np.float64
    for b in range(2):
        ref = sl.solve_triangular(L[b].astype(t), t(alpha) * B[b].astype(t), lower=True)
        tol = 1e-13 if dtype in ("f64", "c128") else 2 * EPS[dtype]
        assert rel_fro(X[b], ref) <= tol


# ---------------------------------------------------------------- conventions
@pytest.mark.parametrize("dtype", DTYPES)
def test_layouts_agree_bitwise(oracle_mod, dtype):
    L, B = ti.generate(dtype, 50, 7, batch=3, kind="solve_tri")
    Xc, _, _ = oracle_solve(oracle_mod, dtype, L, B, 1.0, layout="col")
    Xr, _, _ = oracle_solve(oracle_mod, dtype, L, B, 1.0, layout="row")
    np.testing.assert_array_equal(Xc, Xr)


def test_column_subset_matches_full_solve(oracle_mod):
    L, B = ti.generate("f64", 90, 40, batch=2, kind="dd64")
    Xf, _, _ = oracle_solve(oracle_mod, "f64", L, B, 1.5)
    cols = np.array([0, 3, 17, 39])
    Xs, _, _ = oracle_solve(oracle_mod, "f64", L, B, 1.5, cols=cols)
    np.testing.assert_array_equal(Xs[:, :, cols], Xf[:, :, cols])
    others = np.setdiff1d(np.arange(40), cols)
    np.testing.assert_array_equal(Xs[:, :, others], B[:, :, others])


def test_thread_count_does_not_change_result(oracle_mod):
    L, B = ti.generate("c64", 64, 64, batch=16, kind="dd64")
    X1, _, _ = oracle_solve(oracle_mod, "c64", L, B, 1.0, nthreads=1)
    X4, _, _ = oracle_solve(oracle_mod, "c64", L, B, 1.0, nthreads=4)
    np.testing.assert_array_equal(X1, X4)
