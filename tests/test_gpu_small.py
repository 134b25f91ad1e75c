"""GPU parity of the small-regime path (m <= 64) against the oracle, through
the C ABI, on the workloads' own seeded inputs and on edge cases."""
import os

import numpy as np
import pytest

import trsm_inputs as ti
from gpu_util import (TOL, assert_padding_untouched, assert_parity, gpu_solve_buffers, logical,
                      oracle_buffers, per_system_rel_fro, storage_pair)

pytestmark = pytest.mark.gpu
DTYPES = ["f32", "f64", "c64", "c128"]


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    tg.load_library()
    return dict(torch=torch, tg=tg, oracle=oracle_mod)


def _parity(env, dtype, L, B, alpha, label, single=False, cols=None, **geo_kw):
    a, b, geo = storage_pair(L, B, **geo_kw)
    raw = gpu_solve_buffers(dtype, a, b, geo, alpha, env["torch"], env["tg"], single=single)
    ref = oracle_buffers(dtype, a, b, geo, alpha, env["oracle"], cols=cols)
    assert_padding_untouched(raw, b, geo)
    xg, xr = logical(raw, geo), logical(ref, geo)
    if cols is not None:
        xg, xr = xg[:, :, cols], xr[:, :, cols]
    return assert_parity(dtype, xg, xr, label), xg, xr


# ------------------------------------------------------------- the workloads
def test_solve_tri_8x64x6_matches_oracle_and_golden(env):
    """8 row-major f32 systems, 64 x 64 with 6 RHS (llama.cpp PR 17457's
    test-backend-ops SOLVE_TRI shape)."""
    w = ti.WORKLOADS["solve_tri_8x64x6"]
    L, B = ti.generate("f32", w["m"], w["n"], w["batch"], kind=w["kind"])
    err, xg, _ = _parity(env, "f32", L, B, 1.0, "solve_tri", layout="row")
    path = os.path.join(os.path.dirname(__file__), "golden", "solve_tri_8x64x6_f32.txt")
    rows = [r.split() for r in open(path) if not r.startswith("#")]
    gold = np.array([[float.fromhex(v) for v in r] for r in rows], dtype=np.float32).reshape(8, 64, 6)
    assert float(per_system_rel_fro(xg, gold).max()) <= TOL["f32"]
    # the pull request's own gate: NMSE against the reference below 1e-7
    nmse = float(np.sum((xg.astype(np.float64) - gold) ** 2) / np.sum(gold.astype(np.float64) ** 2))
    assert nmse < 1e-7


@pytest.mark.parametrize("dtype", DTYPES)
def test_square64_single(env, dtype):
    L, B = ti.generate(dtype, 64, 64, 1, kind="dd64")
    _parity(env, dtype, L, B, 1.0, f"square64 {dtype}", single=True)


@pytest.mark.parametrize("dtype", DTYPES)
def test_square64_batch4096(env, dtype):
    L, B = ti.generate(dtype, 64, 64, 4096, kind="dd64")
    _parity(env, dtype, L, B, 1.0, f"square64x4096 {dtype}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("m", [8, 16, 32, 48, 64])
def test_small_sweep_batch16384(env, dtype, m):
    L, B = ti.generate(dtype, m, m, 16384, kind="dd64")
    _parity(env, dtype, L, B, 1.0, f"sweep m={m} {dtype}")


@pytest.mark.parametrize("n", [1, 6, 10, 32])
def test_small_sweep_rectangular(env, n):
    L, B = ti.generate("f32", 64, n, 16384, kind="dd64")
    _parity(env, "f32", L, B, 1.0, f"rect n={n}")


# ------------------------------------------------------------- edge cases
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("m,n", [(1, 1), (1, 9), (5, 3), (17, 10), (33, 7), (63, 65), (64, 130), (40, 2)])
@pytest.mark.parametrize("layout", ["col", "row"])
def test_ragged_shapes_padding_and_alpha(env, dtype, m, n, layout):
    L, B = ti.generate(dtype, m, n, 5, kind="dd64", seed=m * 100 + n)
    alpha = (0.5 - 1.5j) if ti.IS_COMPLEX[dtype] else -1.25
    lda = m + 3
    ldb = (m if layout == "col" else n) + 2
    major_b = n if layout == "col" else m
    _parity(env, dtype, L, B, alpha, f"ragged {dtype} {m}x{n} {layout}", layout=layout, lda=lda,
            ldb=ldb, stride_a=m * lda + 7, stride_b=major_b * ldb + 5)


@pytest.mark.parametrize("n", [10, 3])
def test_non_power_of_two_rhs_count_regression(env, n):
    """llama.cpp PR 17457 met a race only on newer GPUs for 10 RHS (a warp
    count that is not a power of two); run it repeatedly."""
    L, B = ti.generate("f32", 64, n, 4, kind="solve_tri", seed=10)
    for rep in range(20):
        _parity(env, "f32", L, B, 1.0, f"n={n} rep {rep}", layout="row")


@pytest.mark.parametrize("dtype", DTYPES)
def test_alpha_zero_ignores_a(env, dtype):
    torch, tg = env["torch"], env["tg"]
    m, n, batch = 48, 20, 3
    a = torch.full((batch * m * m,), float("nan"), dtype=getattr(torch, {"f32": "float32", "f64": "float64",
                   "c64": "complex64", "c128": "complex128"}[dtype]), device="cuda")
    b = torch.ones(batch * m * n, dtype=a.dtype, device="cuda")
    tg.trsm_llnn_strided_batched(dtype, "col", m, n, 0.0, a, m, m * m, b, m, m * n, batch)
    torch.cuda.synchronize()
    assert bool((b == 0).all())


def test_shared_a_with_zero_stride(env):
    dtype, m, n, batch = "f64", 30, 12, 6
    L, B = ti.generate(dtype, m, n, batch, kind="dd64")
    L[:] = L[0]
    a, b, geo = storage_pair(L[:1], B)
    geo["batch"], geo["sa"] = batch, 0
    b = ti.to_storage(B, "col")
    raw = gpu_solve_buffers(dtype, a, b, geo, 1.0, env["torch"], env["tg"])
    ref = oracle_buffers(dtype, a, b, geo, 1.0, env["oracle"])
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), "shared A")


@pytest.mark.parametrize("dtype", DTYPES)
def test_zero_diagonal_propagates_like_the_oracle(env, dtype):
    L, B = ti.generate(dtype, 40, 16, 2, kind="dd64")
    L[:, 7, 7] = 0
    a, b, geo = storage_pair(L, B)
    raw = gpu_solve_buffers(dtype, a, b, geo, 1.0, env["torch"], env["tg"])
    ref = oracle_buffers(dtype, a, b, geo, 1.0, env["oracle"])
    xg, xr = logical(raw, geo), logical(ref, geo)
    np.testing.assert_array_equal(np.isfinite(xg), np.isfinite(xr))
    fin = np.isfinite(xr)
    assert fin[:, :7].all() and not fin[:, 7:].any()
    assert float(per_system_rel_fro(xg[:, :7], xr[:, :7]).max()) <= TOL[dtype]


def test_solve_convenience_with_torch_layouts(env):
    torch, tg = env["torch"], env["tg"]
    L, B = ti.generate("c64", 24, 5, 3, kind="dd64")
    ref = np.stack([np.linalg.solve(L[i].astype(np.complex128), B[i].astype(np.complex128))
                    for i in range(3)])
    tA = torch.from_numpy(L).cuda()          # row-major (C order) per system
    tB = torch.from_numpy(B.copy()).cuda()
    tg.solve(tA, tB)
    assert float(per_system_rel_fro(tB.cpu().numpy(), ref).max()) <= TOL["c64"]
    tA2 = torch.from_numpy(L).cuda().transpose(1, 2).contiguous().transpose(1, 2)  # column-major
    tB2 = torch.from_numpy(B.copy()).cuda().transpose(1, 2).contiguous().transpose(1, 2)
    tg.solve(tA2, tB2)
    assert float(per_system_rel_fro(tB2.cpu().numpy(), ref).max()) <= TOL["c64"]


@pytest.mark.parametrize("m,n,batch", [(64, 70, 700), (32, 100, 1000), (48, 64, 612), (16, 200, 700)])
def test_persistent_f32_path_many_items(env, m, n, batch):
    """Enough (system, 64-column slice) items for the persistent pipelined
    f32 kernel, with a ragged last slice and items not divisible by the
    warps in flight."""
    L, B = ti.generate("f32", m, n, batch, kind="dd64", seed=m + n)
    _parity(env, "f32", L, B, 0.5, f"pipe m={m} n={n} batch={batch}")


@pytest.mark.parametrize("m", [32, 48, 64])
@pytest.mark.parametrize("geom", ["padded", "gaps", "shared_a"])
def test_persistent_f32_strided_layouts(env, m, geom):
    """Layouts the tensor-copy kernel must describe exactly (or hand to the
    fallback): leading dimensions above m, gaps between systems, and one L
    shared by every system (batch stride 0); the device status word stays
    clear."""
    n, batch = 64, 700
    L, B = ti.generate("f32", m, n, batch, kind="dd64", seed=m)
    kw = {}
    if geom == "padded":
        kw = dict(lda=m + 4, ldb=m + 8)
    elif geom == "gaps":
        kw = dict(stride_a=m * m + 64, stride_b=m * n + 32)
    if geom == "shared_a":
        L[:] = L[0]
        a, b, geo = storage_pair(L[:1], B)
        geo["batch"], geo["sa"] = batch, 0
        b = ti.to_storage(B, "col")
        raw = gpu_solve_buffers("f32", a, b, geo, 1.0, env["torch"], env["tg"])
        ref = oracle_buffers("f32", a, b, geo, 1.0, env["oracle"])
        assert_parity("f32", logical(raw, geo), logical(ref, geo), f"shared A m={m}")
    else:
        _parity(env, "f32", L, B, 1.0, f"{geom} m={m}", **kw)
    assert env["tg"].trsm_device_status() == 0


@pytest.mark.parametrize("dtype", ["f64", "c128"])
@pytest.mark.parametrize("m,n,batch", [(64, 64, 1), (64, 100, 3), (16, 64, 40), (48, 9, 7), (32, 200, 2)])
def test_fp64_few_systems_spread_columns(env, dtype, m, n, batch):
    """FP64 batches too small to fill the GPU: the columns of each system go
    to separate CTAs (slices of 1 to 8 columns, ragged last slice)."""
    L, B = ti.generate(dtype, m, n, batch, kind="dd64", seed=m * n + batch)
    alpha = (0.75 + 0.5j) if ti.IS_COMPLEX[dtype] else 0.75
    _parity(env, dtype, L, B, alpha, f"spread {dtype} m={m} n={n} batch={batch}")


@pytest.mark.parametrize("m,n,batch", [(64, 64, 700), (64, 40, 400), (64, 100, 350), (48, 64, 612), (32, 64, 900),
                                       (64, 32, 700), (48, 17, 500), (32, 30, 800)])
def test_persistent_c64_path_many_items(env, m, n, batch):
    """Enough (system, column-slice) items for the persistent complex64 TMA
    kernel: 64-column slices (a warp pair per item) and, for n <= 32,
    32-column slices (a warp per item); ragged last slices, complex alpha,
    NaN in the upper triangle."""
    L, B = ti.generate("c64", m, n, batch, kind="dd64", seed=3 * m + n)
    _parity(env, "c64", L, B, 0.5 - 0.75j, f"c64 tma m={m} n={n} batch={batch}")
    assert env["tg"].trsm_device_status() == 0


@pytest.mark.parametrize("m", [32, 48, 64])
@pytest.mark.parametrize("geom", ["padded", "gaps", "shared_a"])
def test_persistent_c64_strided_layouts(env, m, geom):
    """The complex64 TMA kernel on layouts its tensor maps must describe:
    padded leading dimensions, gaps between systems, one shared L."""
    n, batch = 64, 700
    L, B = ti.generate("c64", m, n, batch, kind="dd64", seed=m + 1)
    if geom == "shared_a":
        L[:] = L[0]
        a, b, geo = storage_pair(L[:1], B)
        geo["batch"], geo["sa"] = batch, 0
        b = ti.to_storage(B, "col")
        raw = gpu_solve_buffers("c64", a, b, geo, 1.0, env["torch"], env["tg"])
        ref = oracle_buffers("c64", a, b, geo, 1.0, env["oracle"])
        assert_parity("c64", logical(raw, geo), logical(ref, geo), f"shared A m={m}")
    else:
        kw = dict(lda=m + 2, ldb=m + 4) if geom == "padded" else dict(stride_a=m * m + 32, stride_b=m * n + 16)
        _parity(env, "c64", L, B, 1.0, f"{geom} m={m}", **kw)
    assert env["tg"].trsm_device_status() == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("m,n,batch,layout", [
    (8, 8, 16384, "col"),     # the sweep's m = 8 point
    (8, 3, 4096, "row"),      # reciprocals shared from three columns on
    (7, 37, 300, "col"),      # ragged m, odd n: systems straddle CTAs
    (3, 1, 1000, "row"),      # reciprocals per thread
    (5, 2, 3, "col"),
    (1, 300, 2, "row"),
])
def test_tiny_systems(env, dtype, m, n, batch, layout):
    """m <= 8 runs one thread per (system, column): batches up to the
    sweep's 16384, both layouts, padded leading dimensions and gaps between
    systems, complex alpha."""
    L, B = ti.generate(dtype, m, n, batch, kind="dd64", seed=m * 100 + n)
    alpha = (0.75 - 0.5j) if ti.IS_COMPLEX[dtype] else 0.75
    ld_b = (m if layout == "col" else n) + 3
    a, b, geo = storage_pair(L, B, layout=layout, lda=m + 1, ldb=ld_b,
                             stride_a=m * (m + 1) + 8, stride_b=ld_b * (n if layout == "col" else m) + 16)
    raw = gpu_solve_buffers(dtype, a, b, geo, alpha, env["torch"], env["tg"])
    ref = oracle_buffers(dtype, a, b, geo, alpha, env["oracle"])
    assert_padding_untouched(raw, b, geo)
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), f"tiny {dtype} m={m} n={n} {layout}")
