"""Helpers for the GPU parity tests: run the CUDA library through its C ABI
on the same seeded storage the oracle sees, and compare."""
import numpy as np

import trsm_inputs as ti

TOL = {"f32": 1e-5, "c64": 1e-5, "f64": 1e-12, "c128": 1e-12}


def storage_pair(L, B, layout="col", lda=None, ldb=None, stride_a=None, stride_b=None, nan_upper=True):
    """(A buffer, B buffer, geometry) exactly as the oracle helper lays them out."""
    batch, m, _ = L.shape
    n = B.shape[2]
    lda = m if lda is None else lda
    ldb = (m if layout == "col" else n) if ldb is None else ldb
    Lw = L
    if nan_upper and m > 1:
        Lw = L.copy()
        Lw[:, np.triu(np.ones((m, m), dtype=bool), 1)] = np.nan
    a = ti.to_storage(Lw, layout, lda, stride_a)
    b = ti.to_storage(B, layout, ldb, stride_b)
    sa = stride_a if stride_a is not None else m * lda
    sb = stride_b if stride_b is not None else (n if layout == "col" else m) * ldb
    return a, b, dict(m=m, n=n, batch=batch, layout=layout, lda=lda, ldb=ldb, sa=sa, sb=sb)


def gpu_solve_buffers(dtype, a_buf, b_buf, geo, alpha, torch, tg, single=False):
    """Upload, solve with the library, download the raw B buffer."""
    tA = torch.from_numpy(a_buf).cuda()
    tB = torch.from_numpy(b_buf).cuda()
    if single:
        assert geo["batch"] == 1 and geo["layout"] == "col"
        tg.trsm_llnn(dtype, geo["m"], geo["n"], alpha, tA, geo["lda"], tB, geo["ldb"])
    else:
        tg.trsm_llnn_strided_batched(dtype, geo["layout"], geo["m"], geo["n"], alpha, tA, geo["lda"],
                                     geo["sa"], tB, geo["ldb"], geo["sb"], geo["batch"])
    torch.cuda.synchronize()
    return tB.cpu().numpy()


def oracle_buffers(dtype, a_buf, b_buf, geo, alpha, oracle, cols=None):
    out = b_buf.copy()
    oracle.trsm_llnn(dtype, geo["m"], geo["n"], alpha, a_buf, geo["lda"], out, geo["ldb"],
                     layout=geo["layout"], stride_a=geo["sa"], stride_b=geo["sb"],
                     batch=geo["batch"], cols=cols)
    return out


def logical(raw, geo):
    return ti.from_storage(raw, geo["batch"], geo["m"], geo["n"], geo["layout"], geo["ldb"], geo["sb"])


def per_system_rel_fro(x, ref):
    """Relative Frobenius error of every system of a (batch, m, n) pair."""
    t = np.complex128 if np.iscomplexobj(x) or np.iscomplexobj(ref) else np.float64
    d = (x.astype(t) - ref.astype(t)).reshape(x.shape[0], -1)
    r = ref.astype(t).reshape(ref.shape[0], -1)
    num = np.linalg.norm(d, axis=1)
    den = np.linalg.norm(r, axis=1)
    den[den == 0] = 1.0
    return num / den


def assert_parity(dtype, x_gpu, x_ref, label=""):
    errs = per_system_rel_fro(x_gpu, x_ref)
    worst = float(errs.max()) if errs.size else 0.0
    assert np.all(np.isfinite(x_gpu)), f"{label}: non-finite GPU output"
    assert worst <= TOL[dtype], f"{label}: worst-system rel. Frobenius error {worst:.3e} > {TOL[dtype]}"
    return worst


def assert_padding_untouched(raw_gpu, raw_in, geo):
    """Every element of the B buffer outside the logical matrices keeps its
    input value (NaN padding stays NaN)."""
    mask = np.ones(raw_in.shape, dtype=bool)
    idx = ti.to_storage(np.zeros((geo["batch"], geo["m"], geo["n"])), geo["layout"], geo["ldb"],
                        geo["sb"], pad=1.0)
    mask = idx != 0  # padding positions hold 1.0, logical ones 0.0
    a, b = raw_gpu[mask], raw_in[mask]
    same = (a == b) | (np.isnan(a) & np.isnan(b))
    assert np.all(same), "library wrote outside the logical matrices"
