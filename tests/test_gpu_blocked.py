"""GPU parity of the blocked path (m > 64: diagonal-block inversion, block
apply, trailing GEMM update) against the oracle, through the C ABI."""
import numpy as np
import pytest

import trsm_inputs as ti
from gpu_util import (TOL, assert_padding_untouched, assert_parity, gpu_solve_buffers, logical,
                      oracle_buffers, storage_pair)

pytestmark = pytest.mark.gpu
DTYPES = ["f32", "f64", "c64", "c128"]
TORCH_T = {"f32": "float32", "f64": "float64", "c64": "complex64", "c128": "complex128"}


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    tg.load_library()
    return dict(torch=torch, tg=tg, oracle=oracle_mod)


def _ex_solve(env, dtype, L, B, alpha, nb, lda=None, ldb=None, cols=None):
    """Column-major single system through trsm_llnn_ex with a torch workspace."""
    torch, tg = env["torch"], env["tg"]
    a, b, geo = storage_pair(L, B, lda=lda, ldb=ldb, nan_upper=L.shape[1] <= 4096)
    m, n = geo["m"], geo["n"]
    ws_bytes = tg.trsm_llnn_workspace_bytes(dtype, m, n, nb)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    tA = torch.from_numpy(a).cuda()
    tB = torch.from_numpy(b).cuda()
    tg.trsm_llnn_ex(dtype, m, n, alpha, tA, geo["lda"], tB, geo["ldb"], nb, ws, ws_bytes)
    torch.cuda.synchronize()
    raw = tB.cpu().numpy()
    del tA, tB, ws
    ref = oracle_buffers(dtype, a, b, geo, alpha, env["oracle"], cols=cols)
    xg, xr = logical(raw, geo), logical(ref, geo)
    if cols is not None:
        xg, xr = xg[:, :, cols], xr[:, :, cols]
    else:
        assert_padding_untouched(raw, b, geo)
    return xg, xr


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("nb", [128, 256, 512])
@pytest.mark.parametrize("m,n", [(65, 3), (129, 40), (300, 17), (700, 130)])
def test_ragged_blocked(env, dtype, nb, m, n):
    L, B = ti.generate(dtype, m, n, 1, kind="ddm", seed=m + n)
    alpha = (1.5 - 0.5j) if ti.IS_COMPLEX[dtype] else 1.5
    xg, xr = _ex_solve(env, dtype, L, B, alpha, nb, lda=m + 5, ldb=m + 3)
    assert_parity(dtype, xg, xr, f"{dtype} m={m} n={n} nb={nb}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_default_entry_allocates_its_workspace(env, dtype):
    L, B = ti.generate(dtype, 520, 33, 1, kind="ddm")
    a, b, geo = storage_pair(L, B)
    raw = gpu_solve_buffers(dtype, a, b, geo, 2.0, env["torch"], env["tg"], single=True)
    ref = oracle_buffers(dtype, a, b, geo, 2.0, env["oracle"])
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), "trsm_llnn auto workspace")


@pytest.mark.parametrize("dtype", ["f32", "c128"])
@pytest.mark.parametrize("layout", ["col", "row"])
def test_batched_blocked(env, dtype, layout):
    L, B = ti.generate(dtype, 150, 20, 3, kind="ddm")
    a, b, geo = storage_pair(L, B, layout=layout, lda=151, ldb=(150 if layout == "col" else 20) + 1)
    raw = gpu_solve_buffers(dtype, a, b, geo, 0.75, env["torch"], env["tg"])
    ref = oracle_buffers(dtype, a, b, geo, 0.75, env["oracle"])
    assert_padding_untouched(raw, b, geo)
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), f"batched blocked {layout}")


@pytest.mark.parametrize("dtype,m,nb", [
    ("f64", 1000, 256),
    ("f32", 1000, 512),   # doubling: 128-row blocks, then 256 and 512; last block 488 rows
    ("f32", 700, 512),    # last block 188 rows: lower-left blocks past m zeroed
    ("c64", 1536, 256),   # three full blocks
    ("c64", 1000, 512),
    ("f32", 1000, 128),
])
def test_inverse_blocks_times_diagonal_blocks_is_identity(env, dtype, m, nb):
    """The inverted diagonal blocks left in the workspace satisfy W_t D_t = I
    and have a zero upper triangle: the identity-tile substitution with the
    blocked inverse formula (f64), and for f32 / c64 the one-CTA 128-row
    inversion followed by the doubling products, ragged last blocks
    included (padding rows and columns are identity)."""
    torch, tg = env["torch"], env["tg"]
    n = 16   # past the few-right-hand-side path
    L, B = ti.generate(dtype, m, n, 1, kind="ddm")
    a, b, geo = storage_pair(L, B)
    ws_bytes = tg.trsm_llnn_workspace_bytes(dtype, m, n, nb)
    ws = torch.full((ws_bytes,), 0xFF, dtype=torch.uint8, device="cuda")   # NaN until written
    tA, tB = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    tg.trsm_llnn_ex(dtype, m, n, 1.0, tA, m, tB, m, nb, ws, ws_bytes)
    torch.cuda.synchronize()
    np_t = {"f32": np.float32, "f64": np.float64, "c64": np.complex64, "c128": np.complex128}[dtype]
    W = ws.cpu().numpy().view(np_t)
    atol = 1e-13 if dtype == "f64" else 2e-5
    for t in range((m + nb - 1) // nb):
        r0, mb = t * nb, min(nb, m - t * nb)
        Wfull = W[t * nb * nb:(t + 1) * nb * nb].reshape(nb, nb).T   # column-major block
        Wt = Wfull[:mb, :mb]
        Dt = L[0, r0:r0 + mb, r0:r0 + mb]
        np.testing.assert_allclose(Wt @ Dt, np.eye(mb), atol=atol, err_msg=f"{dtype} m={m} nb={nb} t={t}")
        assert np.all(np.triu(Wfull, 1) == 0)   # written as zeros, not left over


@pytest.mark.parametrize("dtype", ["f64", "c128", "f32"])
def test_profile_reports_the_three_phases(env, dtype):
    torch, tg = env["torch"], env["tg"]
    m = n = 1024
    L, B = ti.generate(dtype, m, n, 1, kind="ddm")
    a, b, geo = storage_pair(L, B, nan_upper=False)
    ws_bytes = tg.trsm_llnn_workspace_bytes(dtype, m, n, 256)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    tA, tB = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ms = tg.trsm_llnn_profile(dtype, m, n, 1.5, tA, m, tB, m, 256, ws, ws_bytes)
    assert all(v > 0 for v in ms)
    ref = oracle_buffers(dtype, a, b, geo, 1.5, env["oracle"])
    assert_parity(dtype, logical(tB.cpu().numpy(), geo), logical(ref, geo), "profile entry")


# ------------------------------------------------------------- full workloads
@pytest.mark.parametrize("dtype", ["f64", "c128"])
@pytest.mark.parametrize("m", [1024, 2048, 8192])
@pytest.mark.parametrize("nb", [128, 256, 512])
def test_large_fp64_workload(env, dtype, m, nb):
    """Square m = n, alpha = 1.5, L strictly lower U(-1,1)/m, diagonal 1 + U(0,1);
    every NB of the sweep.  m >= 2048 is checked on the 64 sampled columns."""
    L, B = ti.generate(dtype, m, m, 1, kind="ddm")
    cols = ti.sample_columns(m) if m >= 2048 else None
    xg, xr = _ex_solve(env, dtype, L, B, 1.5, nb, cols=cols)
    assert_parity(dtype, xg, xr, f"{dtype} m={m} nb={nb}")


@pytest.mark.parametrize("dtype", ["f32", "c64"])
def test_large_fp32_workload(env, dtype):
    """Square m = n = 16384 with the table's NB, checked on the 64 sampled columns."""
    m = 16384
    L, B = ti.generate(dtype, m, m, 1, kind="ddm")
    cols = ti.sample_columns(m)
    xg, xr = _ex_solve(env, dtype, L, B, 1.0, 0, cols=cols)
    assert env["tg"].trsm_device_status() == 0
    assert_parity(dtype, xg, xr, f"{dtype} m={m}")


@pytest.mark.parametrize("dtype", ["f32", "c64"])
@pytest.mark.parametrize("nb", [128, 256, 512])
@pytest.mark.parametrize("m,n", [(1000, 777), (1500, 300), (2100, 1030)])
def test_tensor_core_products_ragged(env, dtype, nb, m, n):
    """Shapes that take the tcgen05 (3xTF32) products -- the f32 apply and
    update, the c64 update in real form with a complex beta at t = 0 --:
    ragged row and column tiles, every block size, blocks that fall back to
    the FMA-pipe kernels; the device status word stays clear (no bounded
    wait expired)."""
    L, B = ti.generate(dtype, m, n, 1, kind="ddm", seed=m + 3 * n)
    alpha = (-0.5 + 0.75j) if ti.IS_COMPLEX[dtype] else -0.5
    xg, xr = _ex_solve(env, dtype, L, B, alpha, nb, lda=m + 4, ldb=m + 8)
    assert env["tg"].trsm_device_status() == 0
    assert_parity(dtype, xg, xr, f"tc {dtype} m={m} n={n} nb={nb}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("m,n", [(65, 1), (129, 3), (300, 8), (1000, 2), (4096, 1)])
def test_narrow_path(env, dtype, m, n):
    """Few right-hand sides (n <= 8) through the blocked path: short last
    blocks, every type, padded leading dimensions."""
    L, B = ti.generate(dtype, m, n, 1, kind="ddm", seed=m + 17 * n)
    alpha = (1.5 - 0.5j) if ti.IS_COMPLEX[dtype] else 1.5
    xg, xr = _ex_solve(env, dtype, L, B, alpha, 0, lda=m + 3, ldb=m + 1)
    assert env["tg"].trsm_device_status() == 0
    assert_parity(dtype, xg, xr, f"narrow {dtype} m={m} n={n}")


@pytest.mark.parametrize("dtype", ["f32", "f64"])
def test_narrow_path_large(env, dtype):
    """m = 16384, n = 1: a single right-hand side at full size."""
    m = 16384
    L, B = ti.generate(dtype, m, 1, 1, kind="ddm")
    xg, xr = _ex_solve(env, dtype, L, B, 1.0, 0)
    assert env["tg"].trsm_device_status() == 0
    assert_parity(dtype, xg, xr, f"narrow {dtype} m={m}")


@pytest.mark.parametrize("dtype,n", [("f32", 3), ("c64", 1)])
def test_few_rhs_more_block_rows_than_ctas(env, dtype, n):
    """m = 18688: 146 block rows, more than the resident clusters of four
    hold (one CTA per SM), so some CTAs take a second block row and the
    hand-over between neighbours spans passes."""
    m = 18688
    L, B = ti.generate(dtype, m, n, 1, kind="ddm", seed=5)
    alpha = (0.25 - 1.0j) if ti.IS_COMPLEX[dtype] else 0.75
    xg, xr = _ex_solve(env, dtype, L, B, alpha, 0)
    assert env["tg"].trsm_device_status() == 0
    assert_parity(dtype, xg, xr, f"few-rhs multi-pass {dtype} m={m} n={n}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("m,n", [(513, 1), (640, 8), (1000, 2), (2049, 5), (4096, 3)])
def test_few_rhs_persistent_path(env, dtype, m, n):
    """n <= 8 with 16-byte aligned columns of L: the persistent few-right-hand-
    side kernel (one CTA per 128-row block row, each publishing its x_t to
    the CTAs below; for f32 with n > 1 and for c64 in clusters of four whose
    CTAs hand x_t to the next one directly), ragged last block rows (idle
    CTAs in the last cluster), complex alpha, padded leading
    dimensions; the device status word stays clear, and the phase times show
    that this kernel ran (no separate applies; complex128 from five columns
    on takes the blocked path)."""
    torch, tg = env["torch"], env["tg"]
    per16 = {"f32": 4, "f64": 2, "c64": 2, "c128": 1}[dtype]  # elements in 16 bytes
    lda = (m + per16 - 1) // per16 * per16 + per16           # padded, every column 16-byte aligned
    L, B = ti.generate(dtype, m, n, 1, kind="ddm", seed=m + 31 * n)
    alpha = (0.5 + 1.25j) if ti.IS_COMPLEX[dtype] else -1.25
    xg, xr = _ex_solve(env, dtype, L, B, alpha, 0, lda=lda, ldb=m + 3)
    assert tg.trsm_device_status() == 0
    assert_parity(dtype, xg, xr, f"few-rhs {dtype} m={m} n={n}")

    a, b, geo = storage_pair(L, B, lda=lda, ldb=m + 3)
    ws_bytes = tg.trsm_llnn_workspace_bytes(dtype, m, n, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    tA, tB = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ms = tg.trsm_llnn_profile(dtype, m, n, alpha, tA, geo["lda"], tB, geo["ldb"], 0, ws, ws_bytes)
    if dtype == "c128" and n > 4:   # complex128 keeps five or more columns on the blocked path
        assert ms[1] > 0.0, f"blocked {dtype} m={m} n={n}: phases {ms}"
    else:
        assert ms[1] == 0.0 and ms[2] > 0.0, f"few-rhs {dtype} m={m} n={n}: phases {ms}"
    assert_parity(dtype, logical(tB.cpu().numpy(), geo), xr, f"few-rhs profiled {dtype} m={m} n={n}")


@pytest.mark.parametrize("m,n,nb,ld_pad", [
    (512, 256, 256, 0),    # two blocks: one update, then both applies in one launch
    (528, 257, 256, 1),    # 16-row last block, one column past a tile, odd ldb (scalar splits)
    (520, 300, 256, 0),    # 8-row last block: the per-block flow
    (1280, 600, 128, 3),   # ten blocks, ragged column tiles
    (3000, 512, 512, 0),   # 440-row last block
])
@pytest.mark.parametrize("dtype", ["f32", "c64"])
def test_lookahead_flow_edges(env, dtype, m, n, nb, ld_pad):
    """Look-ahead form (update t, the scaled panel L_panel D^-1 of block t+1
    and the apply of block t-1 in one launch; c64 in real form with
    interleaved K): block counts, last-block sizes, column raggedness and
    leading dimensions at its edges, complex alpha."""
    L, B = ti.generate(dtype, m, n, 1, kind="ddm", seed=m + n + nb)
    alpha = (-0.75 + 0.5j) if ti.IS_COMPLEX[dtype] else -0.75
    xg, xr = _ex_solve(env, dtype, L, B, alpha, nb, lda=m + ld_pad, ldb=m + ld_pad)
    assert env["tg"].trsm_device_status() == 0
    assert_parity(dtype, xg, xr, f"look-ahead {dtype} m={m} n={n} nb={nb}")


@pytest.mark.parametrize("dtype", ["f32", "c64"])
def test_batched_blocked_padded_systems(env, dtype):
    """Strided batch of two m = 640 systems (the batched blocked path), with
    padding between systems."""
    m, n, batch = 640, 300, 2
    L, B = ti.generate(dtype, m, n, batch, kind="ddm", seed=7)
    a, b, geo = storage_pair(L, B, lda=m + 4, ldb=m + 8, stride_a=m * (m + 4) + 16, stride_b=n * (m + 8) + 32)
    alpha = (0.5 + 0.25j) if ti.IS_COMPLEX[dtype] else 0.5
    raw = gpu_solve_buffers(dtype, a, b, geo, alpha, env["torch"], env["tg"])
    ref = oracle_buffers(dtype, a, b, geo, alpha, env["oracle"])
    assert env["tg"].trsm_device_status() == 0
    assert_padding_untouched(raw, b, geo)
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), f"batched padded {dtype}")
