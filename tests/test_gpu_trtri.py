"""GPU parity of the exported triangular inverse (trsm_trtri_lower) against
the oracle's solve of L X = I, through the C ABI: every type, the small
regime and the blocked path (FMA-pipe, tensor-core and look-ahead flows),
padded leading dimensions, NaN in the never-read upper triangle of A and in
the output buffer before the call."""
import numpy as np
import pytest

import trsm_inputs as ti
from gpu_util import assert_padding_untouched, assert_parity, logical, oracle_buffers, storage_pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    tg.load_library()
    return dict(torch=torch, tg=tg, oracle=oracle_mod)


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
@pytest.mark.parametrize("m", [1, 7, 64, 65, 300, 1000])
def test_inverse_matches_the_oracle(env, dtype, m):
    torch, tg = env["torch"], env["tg"]
    L, _ = ti.generate(dtype, m, 1, 1, kind="ddm", seed=11 * m)
    eye = np.eye(m, dtype=ti.NUMPY[dtype])[None]
    a, ident, geo = storage_pair(L, eye, lda=m + 3, ldb=m + 5)
    # the output buffer starts as NaN in its logical part (the call must set
    # every element) and NaN padding (which must stay untouched)
    start = ti.to_storage(np.full((1, m, m), np.nan, dtype=ti.NUMPY[dtype]), "col", geo["ldb"])
    tA = torch.from_numpy(a).cuda()
    tI = torch.from_numpy(start).cuda()
    tg.trsm_trtri_lower(dtype, m, tA, geo["lda"], tI, geo["ldb"])
    torch.cuda.synchronize()
    raw = tI.cpu().numpy()
    assert tg.trsm_device_status() == 0
    ref = oracle_buffers(dtype, a, ident, geo, 1.0, env["oracle"])
    xg, xr = logical(raw, geo), logical(ref, geo)
    assert_parity(dtype, xg, xr, f"trtri {dtype} m={m}")
    assert np.all(xg[0][np.triu_indices(m, 1)] == 0), "strictly upper part of the inverse must be zero"
    assert_padding_untouched(raw, start, geo)


@pytest.mark.parametrize("dtype", ["f32", "c64"])
def test_inverse_times_matrix_is_identity(env, dtype):
    """m = 2048 (tensor-core look-ahead): L^-1 L = I to single precision."""
    torch, tg = env["torch"], env["tg"]
    m = 2048
    L, _ = ti.generate(dtype, m, 1, 1, kind="ddm", seed=5)
    tL = torch.from_numpy(np.asfortranarray(L[0])).cuda()
    tX = torch.empty((m, m), dtype=tL.dtype, device="cuda").t()  # column-major storage
    tg.trsm_trtri_lower(dtype, m, tL.t().contiguous().t(), m, tX, m)
    torch.cuda.synchronize()
    X = tX.cpu().numpy().astype(np.complex128 if ti.IS_COMPLEX[dtype] else np.float64)
    Lf = L[0].astype(X.dtype)
    err = np.linalg.norm(X @ Lf - np.eye(m)) / np.sqrt(m)
    assert err < 1e-5, f"|| L^-1 L - I ||_F / sqrt(m) = {err:.3e}"
