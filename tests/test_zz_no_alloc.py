"""trsm_llnn_noalloc -- the entry point for callers that cannot allocate
device memory (a library inside a host application that owns all device
memory through its own pool, or a latency-sensitive path on which
cudaMalloc / cudaFree must not run) -- gives the same X as the allocating
entry point trsm_llnn, within the parity tolerances, on consecutive calls
that share its fixed device workspace.

Called through the C ABI with ctypes.  Kept in a file of its own that pytest
collects last; it builds and loads the library itself, so it also passes
alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import trsm_inputs as ti
from gpu_util import TOL, per_system_rel_fro

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 * 1024 * 1024  # TRSM_NOALLOC_SCRATCH_BYTES
ERR_WORKSPACE = 900


@pytest.fixture(scope="module")
def env():
    import torch

    import triangular_solve_gb300 as tg
    from triangular_solve_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    lib = tg.load_library()
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    for name in ("trsm_llnn", "trsm_llnn_noalloc"):
        fn = getattr(lib, name)
        fn.argtypes = [ctypes.c_int, i64, i64, vp, vp, i64, vp, i64, vp]
        fn.restype = ctypes.c_int
    lib.trsm_llnn_workspace_bytes.argtypes = [ctypes.c_int, i64, i64, i64]
    lib.trsm_llnn_workspace_bytes.restype = ctypes.c_size_t
    return dict(torch=torch, lib=lib)


CODE = {"f32": 0, "f64": 1, "c64": 2, "c128": 3}


def _alpha(dtype, a):
    if dtype == "f32":
        return ctypes.byref(ctypes.c_float(a.real))
    if dtype == "f64":
        return ctypes.byref(ctypes.c_double(a.real))
    if dtype == "c64":
        return ctypes.byref((ctypes.c_float * 2)(a.real, a.imag))
    return ctypes.byref((ctypes.c_double * 2)(a.real, a.imag))


def _run(env, fn_name, dtype, L, B, alpha, lda, ldb):
    """One solve through the named C entry point on fresh device copies."""
    torch = env["torch"]
    m, n = B.shape
    a = ti.to_storage(L[None], "col", lda)
    b = ti.to_storage(B[None], "col", ldb)
    tA = torch.from_numpy(a).cuda()
    tB = torch.from_numpy(b).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    rc = getattr(env["lib"], fn_name)(CODE[dtype], m, n, _alpha(dtype, complex(alpha)), tA.data_ptr(),
                                      lda, tB.data_ptr(), ldb, stream)
    assert rc == 0, f"{fn_name} returned {rc}"
    torch.cuda.synchronize()
    return ti.from_storage(tB.cpu().numpy(), 1, m, n, "col", ldb)[0]


# Two consecutive calls per type, the second of a different size, so the
# second call starts from the first call's leftovers in the shared array.
CASES = [(700, 50, 1.5), (333, 90, -0.75)]


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
def test_noalloc_matches_allocating_entry_on_consecutive_calls(env, dtype):
    for i, (m, n, alpha) in enumerate(CASES):
        need = env["lib"].trsm_llnn_workspace_bytes(CODE[dtype], m, n, 0)
        assert 0 < need <= SCRATCH_BYTES
        L, B = ti.generate(dtype, m, n, 1, kind="ddm", seed=40 + i)
        al = complex(alpha, 0.25) if ti.IS_COMPLEX[dtype] else alpha
        ref = _run(env, "trsm_llnn", dtype, L[0], B[0], al, m + 1, m + 3)
        got = _run(env, "trsm_llnn_noalloc", dtype, L[0], B[0], al, m + 1, m + 3)
        assert np.all(np.isfinite(got))
        err = float(per_system_rel_fro(got[None], ref[None])[0])
        assert err <= TOL[dtype], f"call {i + 1}: {dtype} m={m} n={n} rel. error {err:.3e}"


def test_noalloc_small_regime_needs_no_workspace(env):
    L, B = ti.generate("f32", 64, 64, 1, kind="dd64")
    ref = _run(env, "trsm_llnn", "f32", L[0], B[0], 1.0, 64, 64)
    got = _run(env, "trsm_llnn_noalloc", "f32", L[0], B[0], 1.0, 64, 64)
    assert float(per_system_rel_fro(got[None], ref[None])[0]) <= TOL["f32"]


def test_noalloc_rejects_problems_beyond_its_array(env):
    torch = env["torch"]
    # complex128, m = n = 16384: the two X panels alone (2 x NB x n x 16 bytes)
    # exceed the 32 MiB array for every block size, so the call must be
    # rejected before anything is launched (the buffers below are tiny)
    m = n = 16384
    need = env["lib"].trsm_llnn_workspace_bytes(CODE["c128"], m, n, 0)
    assert need > SCRATCH_BYTES
    a = torch.zeros(1, dtype=torch.complex128, device="cuda")
    rc = env["lib"].trsm_llnn_noalloc(CODE["c128"], m, n, _alpha("c128", 1 + 0j), a.data_ptr(), m,
                                      a.data_ptr(), m, torch.cuda.current_stream().cuda_stream)
    assert rc == ERR_WORKSPACE
