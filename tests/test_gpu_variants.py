"""GPU parity of every TRSM variant (trsm_general: side, triangle, op, unit
diagonal) against the oracle's general solve, through the C ABI: each type,
shapes that send the mapped solve through the small regime, the blocked
path and (f32 / c64) the tensor-core look-ahead; padded leading dimensions,
NaN in every entry of A the variant must not read and in B's padding (left
untouched)."""
import itertools

import numpy as np
import pytest

import trsm_inputs as ti
from gpu_util import TOL, assert_parity

pytestmark = pytest.mark.gpu
VARIANTS = ["".join(v) for v in itertools.product("LR", "LU", "NTC", "NU")]


@pytest.fixture(scope="module")
def env(oracle_mod):
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    tg.load_library()
    return dict(torch=torch, tg=tg, oracle=oracle_mod)


def _case(dtype, variant, m, n, seed):
    side, uplo, _, diag = variant
    rng = np.random.default_rng(seed)
    k = m if side == "L" else n
    cplx = ti.IS_COMPLEX[dtype]

    def u(shape):
        x = rng.uniform(-1, 1, shape)
        return x + 1j * rng.uniform(-1, 1, shape) if cplx else x

    A = u((k, k)) / k
    A[np.diag_indices(k)] = (1 + rng.uniform(0, 1, k)) + (1j * (1 + rng.uniform(0, 1, k)) if cplx else 0)
    unread = np.triu_indices(k, 1) if uplo == "L" else np.tril_indices(k, -1)
    A[unread] = np.nan
    if diag == "U":
        A[np.diag_indices(k)] = np.nan
    B = u((m, n))
    lda, ldb = k + 3, m + 2
    a = ti.to_storage(A.astype(ti.NUMPY[dtype])[None], "col", lda)
    b = ti.to_storage(B.astype(ti.NUMPY[dtype])[None], "col", ldb)
    return a, b, k, lda, ldb


def _run(env, dtype, variant, m, n, seed):
    torch, tg = env["torch"], env["tg"]
    a, b, k, lda, ldb = _case(dtype, variant, m, n, seed)
    alpha = (0.5 - 0.75j) if ti.IS_COMPLEX[dtype] else -0.5
    tA, tB = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    side, uplo, trans, diag = variant
    tg.trsm_general(dtype, side, uplo, trans, diag, m, n, alpha, tA, lda, tB, ldb)
    torch.cuda.synchronize()
    raw = tB.cpu().numpy()
    assert tg.trsm_device_status() == 0
    ref = b.copy()
    env["oracle"].trsm_general(dtype, side, uplo, trans, diag, m, n, alpha, a, lda, ref, ldb)
    xg = ti.from_storage(raw, 1, m, n, "col", ldb)
    xr = ti.from_storage(ref, 1, m, n, "col", ldb)
    assert_parity(dtype, xg, xr, f"{variant} {dtype} m={m} n={n}")
    pad = ti.to_storage(np.zeros((1, m, n)), "col", ldb, pad=1.0) != 0
    assert np.all(np.isnan(raw[pad])), "B's padding must stay untouched"


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
@pytest.mark.parametrize("m,n", [(17, 9), (64, 40), (200, 130)])
@pytest.mark.parametrize("variant", VARIANTS)
def test_variant_matches_the_oracle(env, variant, dtype, m, n):
    _run(env, dtype, variant, m, n, seed=m * 31 + n + VARIANTS.index(variant))


@pytest.mark.parametrize("dtype", ["f32", "c64"])
@pytest.mark.parametrize("variant", VARIANTS)
def test_variant_on_the_tensor_core_path(env, variant, dtype):
    """m = 700, n = 300: the mapped solve has 300+ right-hand sides on either
    side, so it takes the tensor-core look-ahead form."""
    _run(env, dtype, variant, 700, 300, seed=7 + VARIANTS.index(variant))
