"""Backward-error pin on every workload's own seeded inputs:
||L X - alpha B||_F / (||L||_F ||X||_F) <= 1e-6 (f32, c64) and 1e-14 (f64,
c128), with the oracle's X rounded to the storage type.  For m >= 2048 the
check runs on the seeded sample of 64 RHS columns."""
import numpy as np
import pytest

import trsm_inputs as ti
from oracle_util import oracle_solve, residual

BOUND = {"f32": 1e-6, "c64": 1e-6, "f64": 1e-14, "c128": 1e-14}


def _subset(batch, count=256, seed=2):
    if batch <= count:
        return np.arange(batch)
    return np.sort(np.random.default_rng(seed).choice(batch, count, replace=False))


def _check(oracle_mod, dtype, m, n, batch, kind, alpha, layout="col"):
    L, B = ti.generate(dtype, m, n, batch, kind=kind)
    sel = _subset(batch)
    L, B = L[sel], B[sel]
    cols = ti.sample_columns(n) if m >= 2048 else None
    if cols is not None:
        B = np.ascontiguousarray(B[:, :, cols])
    X, _, _ = oracle_solve(oracle_mod, dtype, L, B, alpha, layout=layout,
                           pad_a=np.nan if m <= 1024 else None)
    r = residual(L, X, B, alpha)
    assert r <= BOUND[dtype], (dtype, m, n, r)
    return r


def test_solve_tri_8x64x6(oracle_mod):
    w = ti.WORKLOADS["solve_tri_8x64x6"]
    _check(oracle_mod, "f32", w["m"], w["n"], w["batch"], w["kind"], w["alpha"], w["layout"])


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
@pytest.mark.parametrize("batch", [1, 4096])
def test_square64(oracle_mod, dtype, batch):
    _check(oracle_mod, dtype, 64, 64, batch, "dd64", 1.0)


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
@pytest.mark.parametrize("m", [8, 16, 32, 48, 64])
def test_small_sweep(oracle_mod, dtype, m):
    _check(oracle_mod, dtype, m, m, 16384, "dd64", 1.0)


@pytest.mark.parametrize("n", [1, 6, 10, 32])
def test_small_sweep_rectangular(oracle_mod, n):
    _check(oracle_mod, "f32", 64, n, 16384, "dd64", 1.0)


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["f64", "c128"])
@pytest.mark.parametrize("m", [1024, 2048, 8192])
def test_large_fp64(oracle_mod, dtype, m):
    _check(oracle_mod, dtype, m, m, 1, "ddm", 1.5)


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["f32", "c64"])
def test_large_fp32(oracle_mod, dtype):
    _check(oracle_mod, dtype, 16384, 16384, 1, "ddm", 1.0)


def test_golden_solve_tri_8x64x6_still_reproduced(oracle_mod):
    """The stored expected values of the 8 x 64 x 6 workload still match."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "solve_tri_8x64x6_f32.txt")
    rows = [l.split() for l in open(path) if not l.startswith("#")]
    gold = np.array([[float.fromhex(v) for v in r] for r in rows], dtype=np.float32)
    L, B = ti.generate("f32", 64, 6, 8, kind="solve_tri")
    X, _, _ = oracle_solve(oracle_mod, "f32", L, B, 1.0, layout="row")
    np.testing.assert_array_equal(X.reshape(8 * 64, 6), gold)
