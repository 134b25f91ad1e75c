"""Helpers shared by the oracle and parity tests (layout marshalling only)."""
import numpy as np

import trsm_inputs as ti


def oracle_solve(oracle, dtype, L, B, alpha, *, layout="col", lda=None, ldb=None,
                 stride_a=None, stride_b=None, cols=None, nthreads=0, pad_a=np.nan):
    """Lay out logical L (batch, m, m) and B (batch, m, n), run the oracle,
    return (X logical, raw B buffer, storage geometry)."""
    batch, m, _ = L.shape
    n = B.shape[2]
    lda = m if lda is None else lda
    ldb = (m if layout == "col" else n) if ldb is None else ldb
    Lw = L
    if pad_a is not None and m > 1:
        # NaN in the strictly upper part of A must never reach X
        Lw = L.copy()
        Lw[:, np.triu(np.ones((m, m), dtype=bool), 1)] = np.nan
    a_buf = ti.to_storage(Lw, layout, lda, stride_a, pad=pad_a)
    b_buf = ti.to_storage(B, layout, ldb, stride_b)
    sa = stride_a if stride_a is not None else (m * lda)
    major_b = n if layout == "col" else m
    sb = stride_b if stride_b is not None else major_b * ldb
    oracle.trsm_llnn(dtype, m, n, alpha, a_buf, lda, b_buf, ldb, layout=layout,
                     stride_a=sa, stride_b=sb, batch=batch, cols=cols, nthreads=nthreads)
    X = ti.from_storage(b_buf, batch, m, n, layout, ldb, sb)
    return X, b_buf, dict(ldb=ldb, stride_b=sb)


def rel_fro(x, ref):
    """Relative Frobenius error ||x - ref||_F / ||ref||_F in float64/complex128."""
    x = np.asarray(x).astype(np.complex128 if np.iscomplexobj(x) else np.float64)
    ref = np.asarray(ref).astype(x.dtype)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((x - ref).ravel()) / (den if den else 1.0))


def worst_system_rel_fro(x, ref):
    """Largest per-system relative Frobenius error of a (batch, m, n) pair."""
    return max(rel_fro(x[b], ref[b]) for b in range(x.shape[0]))


def residual(L, X, B, alpha):
    """||L X - alpha B||_F / (||L||_F ||X||_F), per system max, in high precision."""
    worst = 0.0
    cplx = np.iscomplexobj(L) or np.iscomplexobj(X)
    t = np.complex128 if cplx else np.float64
    for b in range(L.shape[0]):
        Lb = L[b].astype(t)
        Xb = X[b].astype(t)
        r = Lb @ Xb - t(alpha) * B[b].astype(t)
        den = np.linalg.norm(Lb) * np.linalg.norm(Xb)
        worst = max(worst, float(np.linalg.norm(r) / (den if den else 1.0)))
    return worst
