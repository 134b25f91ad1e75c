"""GPU parity of batches of medium systems (m = 128), which run in one launch
of the small regime's chunked kernel (L on chip) instead of the blocked path
system by system: every type, batch sizes from 1 to 1024, ragged and full
column counts, padded strides, a shared A, NaN in the never-read upper
triangle and in the padding (left untouched); a misaligned leading
dimension falls back to the blocked path and must agree as well."""
import numpy as np
import pytest

import trsm_inputs as ti
from gpu_util import (assert_padding_untouched, assert_parity, gpu_solve_buffers, logical, oracle_buffers,
                      storage_pair)

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
@pytest.mark.parametrize("n,batch", [(128, 1), (9, 4), (33, 7), (64, 64), (100, 3), (130, 2), (128, 1024)])
def test_medium_batch_matches_the_oracle(env, dtype, n, batch):
    m = 128
    L, B = ti.generate(dtype, m, n, batch, kind="ddm", seed=n + batch)
    pad = {"f32": 4, "f64": 2, "c64": 2, "c128": 1}[dtype]  # keeps every column 16-byte aligned
    lda, ldb = m + pad, m + 2 * pad
    a, b, geo = storage_pair(L, B, lda=lda, ldb=ldb, stride_a=m * lda + 4 * pad, stride_b=n * ldb + 8 * pad)
    alpha = (0.5 - 1.25j) if ti.IS_COMPLEX[dtype] else -1.25
    raw = gpu_solve_buffers(dtype, a, b, geo, alpha, env["torch"], env["tg"])
    ref = oracle_buffers(dtype, a, b, geo, alpha, env["oracle"])
    assert_padding_untouched(raw, b, geo)
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), f"m=128 {dtype} n={n} batch={batch}")


@pytest.mark.parametrize("dtype", ["f32", "c128"])
def test_medium_shared_matrix_and_misaligned_fallback(env, dtype):
    m, n, batch = 128, 40, 5
    L, B = ti.generate(dtype, m, n, batch, kind="ddm", seed=9)
    L[:] = L[0]  # one matrix for every system: strideA = 0
    for lda in (m, m + 1):  # m + 1: columns not 16-byte aligned -> the blocked path
        a, b, geo = storage_pair(L[:1], B, lda=lda, ldb=m + 3, stride_a=0)
        geo["batch"] = batch
        geo["sa"] = 0
        raw = gpu_solve_buffers(dtype, a, b, geo, 1.0, env["torch"], env["tg"])
        ref = oracle_buffers(dtype, a, b, geo, 1.0, env["oracle"])
        assert_parity(dtype, logical(raw, geo), logical(ref, geo), f"m=128 {dtype} lda={lda}")
