"""GPU parity of the batched blocked path: strided batches of m > 64 systems
solved by one launch sequence over the whole batch (the inversion, then per
block row one apply, one trailing update and one copy back, each kernel
carrying the system index in its grid), against the oracle, through the C
ABI.  Every type; ragged orders and column counts across block sizes;
column- and row-major; padded leading dimensions and gaps between systems;
one A shared by every system (strideA = 0); NaN in the never-read upper
triangle and in the padding, which must stay untouched."""
import numpy as np
import pytest

import trsm_inputs as ti
from gpu_util import (assert_padding_untouched, assert_parity, gpu_solve_buffers, logical, oracle_buffers,
                      storage_pair)

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


def _alpha(dtype):
    return (0.75 - 0.5j) if ti.IS_COMPLEX[dtype] else -0.75


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("m,n,batch", [(65, 3, 5), (129, 40, 3), (200, 17, 8), (256, 256, 6), (300, 1, 4),
                                       (513, 70, 3)])
@pytest.mark.parametrize("layout", ["col", "row"])
def test_batched_blocked_matches_the_oracle(env, dtype, m, n, batch, layout):
    L, B = ti.generate(dtype, m, n, batch, kind="ddm", seed=m + 3 * n + batch)
    lda = m + 3
    ldb = (m if layout == "col" else n) + 5
    major_b = n if layout == "col" else m
    a, b, geo = storage_pair(L, B, layout=layout, lda=lda, ldb=ldb, stride_a=m * lda + 7,
                             stride_b=major_b * ldb + 11)
    alpha = _alpha(dtype)
    raw = gpu_solve_buffers(dtype, a, b, geo, alpha, env["torch"], env["tg"])
    ref = oracle_buffers(dtype, a, b, geo, alpha, env["oracle"])
    assert env["tg"].trsm_device_status() == 0
    assert_padding_untouched(raw, b, geo)
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), f"batched {dtype} {layout} m={m} n={n} b={batch}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("layout", ["col", "row"])
def test_batched_blocked_shared_matrix(env, dtype, layout):
    """strideA = 0: every system reads the same A (inverted once)."""
    m, n, batch = 300, 33, 7
    L, B = ti.generate(dtype, m, n, batch, kind="ddm", seed=21)
    L[:] = L[0]
    ldb = (m if layout == "col" else n) + 2
    a, b, geo = storage_pair(L[:1], B, layout=layout, lda=m + 1, ldb=ldb, stride_a=0)
    geo["batch"], geo["sa"] = batch, 0
    alpha = _alpha(dtype)
    raw = gpu_solve_buffers(dtype, a, b, geo, alpha, env["torch"], env["tg"])
    ref = oracle_buffers(dtype, a, b, geo, alpha, env["oracle"])
    assert_padding_untouched(raw, b, geo)
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), f"shared A {dtype} {layout}")


@pytest.mark.parametrize("dtype", ["f32", "c128"])
def test_batched_blocked_many_systems(env, dtype):
    """A large batch of m = 256 systems (the workload the batched path is
    for), contiguous, alpha = 1."""
    m, n, batch = 256, 256, 512
    L, B = ti.generate(dtype, m, n, batch, kind="ddm", seed=5)
    a, b, geo = storage_pair(L, B)
    raw = gpu_solve_buffers(dtype, a, b, geo, 1.0, env["torch"], env["tg"])
    ref = oracle_buffers(dtype, a, b, geo, 1.0, env["oracle"])
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), f"many {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "c64"])
def test_batched_blocked_misaligned_rows(env, dtype):
    """Leading dimensions that are not a multiple of 16 bytes: the single-
    precision products fall back to the generic GEMM kernel."""
    m, n, batch = 190, 21, 4
    L, B = ti.generate(dtype, m, n, batch, kind="ddm", seed=8)
    a, b, geo = storage_pair(L, B, lda=m + 1, ldb=m + 1, stride_a=m * (m + 1) + 1, stride_b=n * (m + 1) + 1)
    alpha = _alpha(dtype)
    raw = gpu_solve_buffers(dtype, a, b, geo, alpha, env["torch"], env["tg"])
    ref = oracle_buffers(dtype, a, b, geo, alpha, env["oracle"])
    assert_padding_untouched(raw, b, geo)
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), f"misaligned {dtype}")
