"""Seeded synthetic inputs for the TRSM workloads (numpy only).

This module is shared by the oracle tests, the CUDA parity tests and the
benchmark.  It draws random numbers and lays values out in memory; it holds
none of the solve's arithmetic and imports neither the oracle nor the CUDA
library.

Recipe (every instance starts from a fresh ``numpy.random.default_rng(seed)``,
seed 0 unless stated):

* draws, in this order, each one float64 array of uniforms in [0, 1) in
  logical (batch, row, col) C-order:  L_re, [L_im], B_re, [B_im]
  (the imaginary draws only for complex types);
* L: the strictly upper part is zero; the strictly lower part and the
  diagonal are mapped from the same draw by the workload's ``kind``:

  - ``"solve_tri"``  strictly lower U(-0.1, 0.1), diagonal U(1, 2)
    (the batched 8 x (64 x 64, 6 right-hand sides) shape benchmarked in the
    llama.cpp SOLVE_TRI pull request, its test-backend-ops line);
  - ``"dd64"``       strictly lower U(-1, 1)/64, diagonal 1 + U(0, 1);
  - ``"ddm"``        strictly lower U(-1, 1)/m,  diagonal 1 + U(0, 1);

  for complex types the real and imaginary parts are drawn independently
  from the same real distribution;
* B: U(-1, 1) (each part, for complex);
* values are cast to the storage type before being laid out, so the logical
  values do not depend on the layout.

For m >= 2048 parity and the CPU baseline use a seeded sample of 64 RHS
columns: ``default_rng(1).choice(n, 64, replace=False)``, sorted.
"""
from __future__ import annotations

import numpy as np

NUMPY = {"f32": np.float32, "f64": np.float64, "c64": np.complex64, "c128": np.complex128}
IS_COMPLEX = {"f32": False, "f64": False, "c64": True, "c128": True}
ELEM_BYTES = {"f32": 4, "f64": 8, "c64": 8, "c128": 16}


def _map_l(u: np.ndarray, kind: str, m: int) -> np.ndarray:
    """Map a (batch, m, m) uniform draw to L's values in place (upper -> 0)."""
    diag = u.diagonal(axis1=1, axis2=2).copy()
    if kind == "solve_tri":
        u *= 0.2
        u -= 0.1
        dvals = 1.0 + diag
    elif kind in ("dd64", "ddm"):
        scale = 64.0 if kind == "dd64" else float(m)
        u *= 2.0
        u -= 1.0
        u /= scale
        dvals = 1.0 + diag
    else:
        raise ValueError(f"unknown L kind {kind!r}")
    # zero the strictly upper triangle, one contiguous row tail at a time
    for i in range(m - 1):
        u[:, i, i + 1:] = 0.0
    idx = np.arange(m)
    u[:, idx, idx] = dvals
    return u


def generate(dtype: str, m: int, n: int, batch: int = 1, kind: str = "dd64", seed: int = 0):
    """Return logical ``(L, B)`` of shapes (batch, m, m) and (batch, m, n).

    ``L`` has a zero strictly upper triangle; both are in the storage type.
    """
    rng = np.random.default_rng(seed)
    cplx = IS_COMPLEX[dtype]
    t = NUMPY[dtype]
    l_re = _map_l(rng.random((batch, m, m)), kind, m)
    if cplx:
        l_im = _map_l(rng.random((batch, m, m)), kind, m)
        L = np.empty((batch, m, m), dtype=t)
        L.real = l_re
        L.imag = l_im
        del l_im
    else:
        L = l_re.astype(t, copy=False)
    del l_re
    b_re = rng.random((batch, m, n))
    b_re *= 2.0
    b_re -= 1.0
    if cplx:
        b_im = rng.random((batch, m, n))
        b_im *= 2.0
        b_im -= 1.0
        B = np.empty((batch, m, n), dtype=t)
        B.real = b_re
        B.imag = b_im
    else:
        B = b_re.astype(t, copy=False)
    return L, B


def sample_columns(n: int, count: int = 64, seed: int = 1) -> np.ndarray:
    """Seeded, sorted sample of RHS column indices (all columns if n <= count)."""
    if n <= count:
        return np.arange(n, dtype=np.int64)
    return np.sort(np.random.default_rng(seed).choice(n, count, replace=False)).astype(np.int64)


def to_storage(X: np.ndarray, layout: str = "col", ld: int | None = None,
               stride: int | None = None, pad=None) -> np.ndarray:
    """Lay a logical (batch, rows, cols) array out as a flat strided buffer.

    Column-major: element (r, c) of system b sits at ``b*stride + c*ld + r``;
    row-major: at ``b*stride + r*ld + c``.  Padding (ld beyond the logical
    extent, stride beyond one matrix) is filled with ``pad`` (NaN by default
    for floating types) so that a solver reading it shows up in the result.
    """
    batch, rows, cols = X.shape
    if layout == "col":
        major, minor = cols, rows
        src = X.transpose(0, 2, 1)
    elif layout == "row":
        major, minor = rows, cols
        src = X
    else:
        raise ValueError(layout)
    ld = minor if ld is None else ld
    if ld < max(1, minor):
        raise ValueError("leading dimension too small")
    stride = major * ld if stride is None else stride
    if batch > 1 and stride < major * ld:
        raise ValueError("batch stride too small")
    fill = np.nan if pad is None else pad
    # every system's extent: (batch-1)*stride + major*ld (stride 0: one matrix shared by the batch)
    size = max(batch * stride, (batch - 1) * stride + major * ld, 1)
    buf = np.full(size, fill, dtype=X.dtype)
    if batch * major * minor:
        view = np.lib.stride_tricks.as_strided(
            buf, shape=(batch, major, minor),
            strides=(stride * buf.itemsize, ld * buf.itemsize, buf.itemsize))
        view[...] = src
    return buf


def from_storage(buf: np.ndarray, batch: int, rows: int, cols: int, layout: str = "col",
                 ld: int | None = None, stride: int | None = None) -> np.ndarray:
    """Inverse of :func:`to_storage`: read a logical (batch, rows, cols) copy."""
    major, minor = (cols, rows) if layout == "col" else (rows, cols)
    ld = minor if ld is None else ld
    stride = major * ld if stride is None else stride
    view = np.lib.stride_tricks.as_strided(
        buf, shape=(batch, major, minor),
        strides=(stride * buf.itemsize, ld * buf.itemsize, buf.itemsize))
    out = np.array(view)
    return out.transpose(0, 2, 1).copy() if layout == "col" else out


def flops(dtype: str, m: int, n: int, batch: int = 1) -> float:
    """Credited work: m^2 n real flops per system, times 4 for complex types."""
    return float(batch) * m * m * n * (4.0 if IS_COMPLEX[dtype] else 1.0)


def algorithmic_bytes(dtype: str, m: int, n: int, batch: int = 1) -> float:
    """Read L's lower triangle once, read B, write X."""
    return float(batch) * ELEM_BYTES[dtype] * (m * (m + 1) / 2 + 2.0 * m * n)


# Named workloads (sizes and value distributions).
WORKLOADS = {
    # 8 independent row-major systems (batch [4,2] flattened), 64 x 64, 6 RHS
    "solve_tri_8x64x6": dict(dtypes=("f32",), m=64, n=6, batch=8, kind="solve_tri",
                             layout="row", alpha=1.0),
    # one square m = n = 64 system per dtype, and the strided batch of 4096
    "square64": dict(dtypes=("f32", "f64", "c64", "c128"), m=64, n=64, batch=4096,
                     kind="dd64", layout="col", alpha=1.0),
    # small-regime sweep, batch 16384
    "small_sweep": dict(dtypes=("f32", "f64", "c64", "c128"), ms=(8, 16, 32, 48, 64),
                        batch=16384, kind="dd64", layout="col", alpha=1.0,
                        rect_n=(1, 6, 10, 32)),
    # large blocked f64 / c128
    "large_fp64": dict(dtypes=("f64", "c128"), ms=(1024, 2048, 8192), kind="ddm",
                       layout="col", alpha=1.5, nbs=(128, 256, 512)),
    # large blocked f32 / c64
    "large_fp32": dict(dtypes=("f32", "c64"), ms=(16384,), kind="ddm", layout="col",
                       alpha=1.0),
}
