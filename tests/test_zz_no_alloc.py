"""trsm_llnn_noalloc -- the entry point for callers that cannot allocate
device memory (a library inside a host application that owns all device
memory through its own pool, or a latency-sensitive path on which
cudaMalloc / cudaFree must not run) -- on consecutive calls that share its
fixed device array:

  * its X matches the allocating entry point trsm_llnn and the oracle, within
    the parity tolerances, on every call of a sequence whose sizes change, so
    each call starts from the previous call's leftovers in the array;
  * the sequence reaches the tensor-core look-ahead paths of f32 and c64,
    whose operand panels and tensor maps then live in the array;
  * once the array is loaded (first call), a call changes neither the
    device's free memory nor torch's caching allocator.

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
CODE = {"f32": 0, "f64": 1, "c64": 2, "c128": 3}


@pytest.fixture(scope="module")
def env(oracle_mod):
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
    lib.trsm_device_status.argtypes = [ctypes.c_int]
    lib.trsm_device_status.restype = ctypes.c_int
    return dict(torch=torch, lib=lib, oracle=oracle_mod)


def _alpha(dtype, a):
    if dtype == "f32":
        return ctypes.byref(ctypes.c_float(a.real))
    if dtype == "f64":
        return ctypes.byref(ctypes.c_double(a.real))
    if dtype == "c64":
        return ctypes.byref((ctypes.c_float * 2)(a.real, a.imag))
    return ctypes.byref((ctypes.c_double * 2)(a.real, a.imag))


class Problem:
    """One system in column-major storage with padded leading dimensions (NaN
    in A's strictly upper part), resident on the device."""

    def __init__(self, env, dtype, m, n, alpha, seed):
        torch = env["torch"]
        L, B = ti.generate(dtype, m, n, 1, kind="ddm", seed=seed)
        self.env, self.dtype, self.m, self.n, self.alpha = env, dtype, m, n, alpha
        self.lda, self.ldb = m + 1, m + 3
        Lw = L.copy()
        Lw[:, np.triu(np.ones((m, m), dtype=bool), 1)] = np.nan
        self.a = ti.to_storage(Lw, "col", self.lda)
        self.b = ti.to_storage(B, "col", self.ldb)
        self.tA = torch.from_numpy(self.a).cuda()
        self.tB0 = torch.from_numpy(self.b).cuda()
        self.tB = self.tB0.clone()

    def call(self, fn_name):
        """Restore B, solve through the named C entry point, return X."""
        torch = self.env["torch"]
        self.tB.copy_(self.tB0)
        torch.cuda.synchronize()
        rc = getattr(self.env["lib"], fn_name)(
            CODE[self.dtype], self.m, self.n, _alpha(self.dtype, complex(self.alpha)), self.tA.data_ptr(),
            self.lda, self.tB.data_ptr(), self.ldb, torch.cuda.current_stream().cuda_stream)
        assert rc == 0, f"{fn_name} returned {rc}"
        torch.cuda.synchronize()
        return ti.from_storage(self.tB.cpu().numpy(), 1, self.m, self.n, "col", self.ldb)[0]

    def oracle(self):
        out = self.b.copy()
        self.env["oracle"].trsm_llnn(self.dtype, self.m, self.n, self.alpha, self.a, self.lda, out, self.ldb)
        return ti.from_storage(out, 1, self.m, self.n, "col", self.ldb)[0]


def _err(x, ref):
    return float(per_system_rel_fro(x[None], ref[None])[0])


# Consecutive calls per type, sizes changing between calls, so every call
# starts from the previous call's leftovers in the shared array.  The f32
# and c64 sequences include a system that takes the tensor-core look-ahead
# form (n >= 256, several block rows), whose operand panels live in the array.
SEQUENCES = {
    "f32": [(700, 50, 1.5), (1024, 1024, 1.0), (333, 90, -0.75)],
    "f64": [(700, 50, 1.5), (333, 90, -0.75)],
    "c64": [(700, 50, 1.5), (768, 512, 0.5), (333, 90, -0.75)],
    "c128": [(700, 50, 1.5), (333, 90, -0.75)],
}


@pytest.mark.parametrize("dtype", ["f32", "f64", "c64", "c128"])
def test_noalloc_matches_allocating_entry_and_oracle_on_consecutive_calls(env, dtype):
    lib = env["lib"]
    for i, (m, n, alpha) in enumerate(SEQUENCES[dtype]):
        # the table's block size, else the largest smaller one, fits the array
        need = min(lib.trsm_llnn_workspace_bytes(CODE[dtype], m, n, nb) for nb in (0, 256, 128))
        assert 0 < need <= SCRATCH_BYTES
        al = complex(alpha, 0.25) if ti.IS_COMPLEX[dtype] else alpha
        p = Problem(env, dtype, m, n, al, seed=40 + i)
        ref = p.call("trsm_llnn")
        orc = p.oracle()
        for rep in range(2):  # the same system twice in a row through the array
            got = p.call("trsm_llnn_noalloc")
            assert np.all(np.isfinite(got))
            e_llnn, e_orc = _err(got, ref), _err(got, orc)
            assert e_llnn <= TOL[dtype], f"call {i + 1}.{rep}: {dtype} m={m} n={n} vs trsm_llnn {e_llnn:.3e}"
            assert e_orc <= TOL[dtype], f"call {i + 1}.{rep}: {dtype} m={m} n={n} vs oracle {e_orc:.3e}"
        assert lib.trsm_device_status(1) == 0


@pytest.mark.parametrize("dtype,m,n", [("f32", 1024, 1024), ("c64", 768, 512), ("f64", 700, 50)])
def test_noalloc_leaves_device_memory_unchanged(env, dtype, m, n):
    torch = env["torch"]
    p = Problem(env, dtype, m, n, 1.0, seed=7)
    p.call("trsm_llnn")
    orc = p.oracle()
    p.call("trsm_llnn_noalloc")  # the array's module and the side stream exist from here on
    stats0 = torch.cuda.memory_stats()
    free0, _ = torch.cuda.mem_get_info()
    got = p.call("trsm_llnn_noalloc")
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0, f"device free memory changed by {free1 - free0} bytes"
    for key in ("reserved_bytes.all.current", "allocated_bytes.all.current", "num_alloc_retries"):
        assert stats1.get(key, 0) == stats0.get(key, 0), key
    assert _err(got, orc) <= TOL[dtype]


def test_noalloc_small_regime_needs_no_workspace(env):
    p = Problem(env, "f32", 64, 64, 1.0, seed=0)
    ref = p.call("trsm_llnn")
    got = p.call("trsm_llnn_noalloc")
    assert _err(got, ref) <= TOL["f32"]
    assert _err(got, p.oracle()) <= TOL["f32"]


def test_noalloc_rejects_problems_beyond_its_array(env):
    torch = env["torch"]
    # complex128, m = n = 16384: the two X panels alone (2 x NB x n x 16 bytes)
    # exceed the 32 MiB array for every block size, so the call must be
    # rejected before anything is launched (the buffers below are tiny)
    m = n = 16384
    need = min(env["lib"].trsm_llnn_workspace_bytes(CODE["c128"], m, n, nb) for nb in (0, 256, 128))
    assert need > SCRATCH_BYTES
    a = torch.zeros(1, dtype=torch.complex128, device="cuda")
    rc = env["lib"].trsm_llnn_noalloc(CODE["c128"], m, n, _alpha("c128", 1 + 0j), a.data_ptr(), m,
                                      a.data_ptr(), m, torch.cuda.current_stream().cuda_stream)
    assert rc == ERR_WORKSPACE
