"""CPU oracle for the left-lower, non-transposed, non-unit TRSM  L X = alpha B,
and for every other TRSM variant (``trsm_general``: side, triangle, op, unit
diagonal; BLAS meaning).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library (``triangular_solve_gb300``) and never serves as its
fallback.

The arithmetic lives in ``trsm_oracle.c`` (plain forward substitution in
double precision, see its header for the passages it follows); this module
only compiles it with the host C compiler and marshals numpy arrays.

Parity status: pinned.  ``tests/test_oracle_pins.py`` checks it against the
identity and diagonal special cases, exact integer recovery, the bidiagonal
and all-ones closed forms, brute-force Gaussian elimination with partial
pivoting on m <= 8, LAPACK's triangular solve, and the backward-error bound
on every workload's inputs.  ``tests/test_oracle_variants.py`` pins the
general variants: a dense library solve of the explicitly formed op(A) for
all 24 variants and four types (NaN in every entry a variant must not read),
bitwise agreement with the left-lower oracle, bidiagonal suffix-sum closed
forms for the left-upper and right-lower cases, and alpha = 0.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# A test that plants a mistake in a temporary copy of the oracle points these
# two variables at that copy and at a scratch build folder.
_SRC = os.environ.get("TRSM_ORACLE_TEST_SRC") or os.path.join(_HERE, "trsm_oracle.c")
_BUILD = os.environ.get("TRSM_ORACLE_TEST_BUILD") or os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f32": 0, "f64": 1, "c64": 2, "c128": 3}
NUMPY = {"f32": np.float32, "f64": np.float64, "c64": np.complex64, "c128": np.complex128}
LAYOUTS = {"col": 0, "row": 1}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_trsm_llnn.argtypes = [
                ctypes.c_int, ctypes.c_int, i64, i64, ctypes.POINTER(ctypes.c_double),
                vp, i64, i64, vp, i64, i64, i64, ctypes.POINTER(ctypes.c_int64), i64,
                ctypes.c_int]
            lib.oracle_trsm_llnn.restype = ctypes.c_int
            lib.oracle_max_threads.restype = ctypes.c_int
            ci = ctypes.c_int
            lib.oracle_trsm_general.argtypes = [ci, ci, ci, ci, ci, i64, i64, ctypes.POINTER(ctypes.c_double),
                                                vp, i64, vp, i64]
            lib.oracle_trsm_general.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def trsm_llnn(dtype: str, m: int, n: int, alpha, A: np.ndarray, lda: int, B: np.ndarray,
              ldb: int, *, layout: str = "col", stride_a: int = 0, stride_b: int = 0,
              batch: int = 1, cols=None, nthreads: int = 0) -> None:
    """Solve in place in ``B`` (a flat or any-shaped C-contiguous numpy buffer).

    ``A`` and ``B`` hold ``batch`` systems laid out with element strides
    ``stride_a`` / ``stride_b`` and leading dimensions ``lda`` / ``ldb`` in
    the given layout, exactly as the CUDA library's strided-batched call reads
    them.  ``cols`` restricts the solve to a subset of RHS columns.
    """
    np_t = NUMPY[dtype]
    if B.dtype != np_t or (A is not None and A.dtype != np_t):
        raise TypeError(f"oracle: arrays must be {np_t}")
    if not B.flags.c_contiguous or (A is not None and not A.flags.c_contiguous):
        raise ValueError("oracle: arrays must be C-contiguous buffers")
    a = complex(alpha)
    al = (ctypes.c_double * 2)(a.real, a.imag)
    if cols is not None:
        cols_arr = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
        cp = cols_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        nc = int(cols_arr.size)
    else:
        cols_arr, cp, nc = None, None, int(n)
    rc = _load().oracle_trsm_llnn(
        DTYPES[dtype], LAYOUTS[layout], int(m), int(n), al,
        None if A is None else A.ctypes.data, int(lda), int(stride_a),
        B.ctypes.data, int(ldb), int(stride_b), int(batch), cp, nc, int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_trsm_llnn: invalid argument {-rc}")


SIDES = {"L": 0, "R": 1}
UPLOS = {"L": 0, "U": 1}
OPS = {"N": 0, "T": 1, "C": 2}
DIAGS = {"N": 0, "U": 1}


def trsm_general(dtype: str, side: str, uplo: str, trans: str, diag: str, m: int, n: int, alpha,
                 A: np.ndarray, lda: int, B: np.ndarray, ldb: int) -> None:
    """Any TRSM variant (BLAS meaning: side L/R, uplo L/U, trans N/T/C, diag
    N/U), column-major, one system, in place in ``B``; see
    ``oracle_trsm_general`` in ``trsm_oracle.c``."""
    np_t = NUMPY[dtype]
    if B.dtype != np_t or (A is not None and A.dtype != np_t):
        raise TypeError(f"oracle: arrays must be {np_t}")
    if not B.flags.c_contiguous or (A is not None and not A.flags.c_contiguous):
        raise ValueError("oracle: arrays must be C-contiguous buffers")
    a = complex(alpha)
    al = (ctypes.c_double * 2)(a.real, a.imag)
    rc = _load().oracle_trsm_general(DTYPES[dtype], SIDES[side], UPLOS[uplo], OPS[trans], DIAGS[diag],
                                     int(m), int(n), al, None if A is None else A.ctypes.data, int(lda),
                                     B.ctypes.data, int(ldb))
    if rc != 0:
        raise ValueError(f"oracle_trsm_general: invalid argument {-rc}")
