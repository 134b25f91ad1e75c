"""trsm_llnn_strided_batched_host -- the strided-batched solve on host
buffers, pipelined in chunks over three internal streams (copy in, solve,
copy out) -- against the oracle,
through the C ABI: chunked batches, row-major systems with gaps between them,
one A shared by all systems, the blocked path, alpha = 0."""
import numpy as np
import pytest

import trsm_inputs as ti
from gpu_util import assert_parity, logical, oracle_buffers, storage_pair

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


def _host_solve(env, dtype, a, b, geo, alpha):
    torch, tg = env["torch"], env["tg"]
    tA = torch.from_numpy(a).pin_memory()
    tB = torch.from_numpy(b.copy()).pin_memory()
    tg.trsm_llnn_strided_batched_host(dtype, geo["layout"], geo["m"], geo["n"], alpha, tA, geo["lda"], geo["sa"],
                                      tB, geo["ldb"], geo["sb"], geo["batch"])
    torch.cuda.synchronize()
    return tB.numpy()


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
@pytest.mark.parametrize("m,n,batch,layout", [(64, 64, 1000, "col"), (48, 20, 37, "row"), (200, 30, 3, "col"),
                                              (7, 5, 2, "col")])
def test_host_entry_matches_oracle(env, dtype, m, n, batch, layout):
    L, B = ti.generate(dtype, m, n, batch, kind="dd64" if m <= 64 else "ddm", seed=m + n + batch)
    minor = m if layout == "col" else n
    major = n if layout == "col" else m
    a, b, geo = storage_pair(L, B, layout=layout, lda=m + 2, ldb=minor + 3, stride_a=m * (m + 2) + 6,
                             stride_b=major * (minor + 3) + 10)
    alpha = (1.25 - 0.5j) if ti.IS_COMPLEX[dtype] else 1.25
    raw = _host_solve(env, dtype, a, b, geo, alpha)
    ref = oracle_buffers(dtype, a, b, geo, alpha, env["oracle"])
    # padding between and inside systems comes back unchanged
    mask = np.ones(b.shape, dtype=bool)
    for s in range(batch):
        for j in range(major):
            o = s * geo["sb"] + j * geo["ldb"]
            mask[o:o + minor] = False
    np.testing.assert_array_equal(raw[mask], b[mask])
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), f"host {dtype} {m}x{n} batch {batch} {layout}")


def test_host_entry_shared_a_and_alpha_zero(env):
    dtype, m, n, batch = "c128", 64, 64, 300
    L, B = ti.generate(dtype, m, n, batch, kind="dd64")
    L[:] = L[0]
    a, b, geo = storage_pair(L[:1], B)
    geo["batch"], geo["sa"] = batch, 0
    b = ti.to_storage(B, "col")
    raw = _host_solve(env, dtype, a, b, geo, 1.0)
    ref = oracle_buffers(dtype, a, b, geo, 1.0, env["oracle"])
    assert_parity(dtype, logical(raw, geo), logical(ref, geo), "host shared A")
    raw0 = _host_solve(env, dtype, np.zeros(1, dtype=a.dtype), b, geo, 0.0)
    assert np.all(raw0 == 0)
