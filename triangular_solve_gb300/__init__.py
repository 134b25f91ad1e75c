"""Python binding of ``libtrsm_gb300.so``, the GB300 (sm_103a) triangular
solver:  L X = alpha B  for X in place of B, L the lower triangle of A
(left side, lower, non-transposed, non-unit diagonal), in f32, f64,
complex64 and complex128.

The functions mirror the C ABI of ``include/trsm.h`` one to one and only
marshal arguments: device pointers come from CUDA torch tensors (or plain
integers), the stream defaults to torch's current stream, and a non-zero
status raises.  Every step of the solve runs in the library's CUDA kernels;
there is no CPU path.  The shared library is built in-tree by
``python -m triangular_solve_gb300.build``; importing this package does not
load it, the first call does (and raises if it was not built).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

__all__ = [
    "trsm_llnn", "trsm_llnn_strided_batched", "trsm_llnn_strided_batched_host", "trsm_llnn_select_nb",
    "trsm_llnn_workspace_bytes", "trsm_llnn_ex", "trsm_llnn_profile", "trsm_general", "trsm_trtri_lower",
    "trsm_status_string", "trsm_llnn_noalloc", "trsm_device_status", "trsm_set_wait_limit",
    "solve", "TrsmError",
    "library_path", "load_library",
]

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libtrsm_gb300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "trsm.h")

DTYPES = {"f32": 0, "f64": 1, "c64": 2, "c128": 3}
LAYOUTS = {"col": 0, "row": 1}
SUCCESS = 0
ERR_WORKSPACE = 900
ERR_CUDA_BASE = 1000

_lock = threading.Lock()
_lib = None


class TrsmError(RuntimeError):
    """A non-zero status from the library."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: status {status}: {trsm_status_string(status)}")


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load the in-tree shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m triangular_solve_gb300.build` "
                "(the solver has no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.trsm_llnn.argtypes = [i32, i64, i64, vp, vp, i64, vp, i64, vp]
        lib.trsm_llnn_strided_batched.argtypes = [i32, i32, i64, i64, vp, vp, i64, i64, vp, i64, i64,
                                                  i64, vp]
        lib.trsm_llnn_strided_batched_host.argtypes = [i32, i32, i64, i64, vp, vp, i64, i64, vp, i64, i64,
                                                       i64, vp]
        lib.trsm_llnn_select_nb.argtypes = [i32, i64, i64]
        lib.trsm_llnn_workspace_bytes.argtypes = [i32, i64, i64, i64]
        lib.trsm_llnn_workspace_bytes.restype = ctypes.c_size_t
        lib.trsm_llnn_ex.argtypes = [i32, i64, i64, vp, vp, i64, vp, i64, i64, vp, ctypes.c_size_t, vp]
        lib.trsm_llnn_profile.argtypes = [i32, i64, i64, vp, vp, i64, vp, i64, i64, vp, ctypes.c_size_t,
                                          vp, ctypes.POINTER(ctypes.c_float)]
        lib.trsm_trtri_lower.argtypes = [i32, i64, vp, i64, vp, i64, vp]
        lib.trsm_general.argtypes = [i32, i32, i32, i32, i32, i64, i64, vp, vp, i64, vp, i64, vp]
        lib.trsm_status_string.argtypes = [i32]
        lib.trsm_status_string.restype = ctypes.c_char_p
        for name in ("trsm_llnn", "trsm_llnn_strided_batched", "trsm_llnn_strided_batched_host", "trsm_llnn_select_nb",
                     "trsm_llnn_ex", "trsm_llnn_profile", "trsm_trtri_lower", "trsm_general"):
            getattr(lib, name).restype = i32
        _lib = lib
        return lib


def declared_functions() -> list[str]:
    """Names of the functions include/trsm.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(trsm_\w+)\s*\(", text, re.M)))


# ------------------------------------------------------------------ marshalling
def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    if isinstance(dtype, str):
        return DTYPES[dtype]
    import torch
    return {torch.float32: 0, torch.float64: 1, torch.complex64: 2, torch.complex128: 3}[dtype]


def _layout_code(layout) -> int:
    return layout if isinstance(layout, int) else LAYOUTS[layout]


def _alpha_buf(code: int, alpha):
    a = complex(alpha)
    if code == 0:
        return ctypes.byref(ctypes.c_float(a.real)), ctypes.c_float
    if code == 1:
        return ctypes.byref(ctypes.c_double(a.real)), ctypes.c_double
    if code == 2:
        return ctypes.byref((ctypes.c_float * 2)(a.real, a.imag)), None
    return ctypes.byref((ctypes.c_double * 2)(a.real, a.imag)), None


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_cuda:
            raise ValueError("the solver takes CUDA (device) tensors; got a CPU tensor")
        return x.data_ptr()
    raise TypeError(f"expected a CUDA tensor or a device pointer, got {type(x)}")


def _stream(stream):
    if stream is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:  # no torch / no device: the legacy default stream
            return 0
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int) -> None:
    if status != SUCCESS:
        raise TrsmError(fn, status)


# ------------------------------------------------------------------ C ABI mirror
def trsm_llnn(dtype, m, n, alpha, A, lda, B, ldb, stream=None) -> None:
    """Single column-major system, in place in B (see include/trsm.h)."""
    code = _dtype_code(dtype)
    al, _ = _alpha_buf(code, alpha)
    _check("trsm_llnn", load_library().trsm_llnn(code, m, n, al, _ptr(A), lda, _ptr(B), ldb,
                                                 _stream(stream)))


_SIDE = {"L": 0, "R": 1}
_UPLO = {"L": 0, "U": 1}
_OP = {"N": 0, "T": 1, "C": 2}
_DIAG = {"N": 0, "U": 1}


def _flag(table, v, what):
    if isinstance(v, str) and v.upper() in table:
        return table[v.upper()]
    if isinstance(v, int) and v in table.values():
        return v
    raise ValueError(f"{what}: {v!r}")


def trsm_general(dtype, side, uplo, trans, diag, m, n, alpha, A, lda, B, ldb, stream=None) -> None:
    """Any TRSM variant, BLAS meaning (side "L"/"R", uplo "L"/"U", trans
    "N"/"T"/"C", diag "N"/"U"), column-major, in place in B (see
    include/trsm.h)."""
    code = _dtype_code(dtype)
    al, _ = _alpha_buf(code, alpha)
    _check("trsm_general", load_library().trsm_general(
        code, _flag(_SIDE, side, "side"), _flag(_UPLO, uplo, "uplo"), _flag(_OP, trans, "trans"),
        _flag(_DIAG, diag, "diag"), m, n, al, _ptr(A), lda, _ptr(B), ldb, _stream(stream)))


def trsm_trtri_lower(dtype, m, A, lda, Ainv, ldinv, stream=None) -> None:
    """Ainv = inverse of the lower triangle of A, both column-major; the
    strictly upper part of Ainv is set to zero (see include/trsm.h)."""
    _check("trsm_trtri_lower", load_library().trsm_trtri_lower(_dtype_code(dtype), m, _ptr(A), lda, _ptr(Ainv),
                                                               ldinv, _stream(stream)))


def trsm_llnn_strided_batched(dtype, layout, m, n, alpha, A, lda, strideA, B, ldb, strideB, batch,
                              stream=None) -> None:
    code = _dtype_code(dtype)
    al, _ = _alpha_buf(code, alpha)
    _check("trsm_llnn_strided_batched", load_library().trsm_llnn_strided_batched(
        code, _layout_code(layout), m, n, al, _ptr(A), lda, strideA, _ptr(B), ldb, strideB, batch,
        _stream(stream)))


def _host_ptr(x):
    if hasattr(x, "data_ptr"):
        if x.is_cuda:
            raise ValueError("trsm_llnn_strided_batched_host takes host (CPU) tensors")
        return x.data_ptr()
    return x


def trsm_llnn_strided_batched_host(dtype, layout, m, n, alpha, A, lda, strideA, B, ldb, strideB, batch,
                                   stream=None) -> None:
    """The strided-batched solve on host buffers (pinned CPU tensors for
    overlapped copies); enqueued on `stream`, B holds X once it has run."""
    code = _dtype_code(dtype)
    al, _ = _alpha_buf(code, alpha)
    _check("trsm_llnn_strided_batched_host", load_library().trsm_llnn_strided_batched_host(
        code, _layout_code(layout), m, n, al, _host_ptr(A), lda, strideA, _host_ptr(B), ldb, strideB, batch,
        _stream(stream)))


def trsm_llnn_select_nb(dtype, m, n) -> int:
    r = load_library().trsm_llnn_select_nb(_dtype_code(dtype), m, n)
    if r < 0:
        raise TrsmError("trsm_llnn_select_nb", r)
    return r


def trsm_llnn_workspace_bytes(dtype, m, n, nb=0) -> int:
    r = load_library().trsm_llnn_workspace_bytes(_dtype_code(dtype), m, n, nb)
    if r == ctypes.c_size_t(-1).value:
        raise ValueError("trsm_llnn_workspace_bytes: invalid arguments")
    return int(r)


def trsm_llnn_ex(dtype, m, n, alpha, A, lda, B, ldb, nb, workspace, ws_bytes, stream=None) -> None:
    code = _dtype_code(dtype)
    al, _ = _alpha_buf(code, alpha)
    _check("trsm_llnn_ex", load_library().trsm_llnn_ex(code, m, n, al, _ptr(A), lda, _ptr(B), ldb, nb,
                                                       _ptr(workspace), ws_bytes, _stream(stream)))


def trsm_llnn_profile(dtype, m, n, alpha, A, lda, B, ldb, nb, workspace, ws_bytes, stream=None):
    """Returns (ms_inversion, ms_apply, ms_update); synchronises the stream."""
    code = _dtype_code(dtype)
    al, _ = _alpha_buf(code, alpha)
    ms = (ctypes.c_float * 3)()
    _check("trsm_llnn_profile", load_library().trsm_llnn_profile(
        code, m, n, al, _ptr(A), lda, _ptr(B), ldb, nb, _ptr(workspace), ws_bytes, _stream(stream), ms))
    return float(ms[0]), float(ms[1]), float(ms[2])


def trsm_llnn_noalloc(dtype, m, n, alpha, A, lda, B, ldb, stream=None) -> None:
    """trsm_llnn that allocates no device memory: the blocked path's workspace
    is a fixed array inside the library (see include/trsm.h).  For callers
    whose host application owns all device memory, or whose path must not
    call cudaMalloc / cudaFree."""
    lib = load_library()
    fn = lib.trsm_llnn_noalloc
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    fn.argtypes = [ctypes.c_int, i64, i64, vp, vp, i64, vp, i64, vp]
    fn.restype = ctypes.c_int
    code = _dtype_code(dtype)
    al, _ = _alpha_buf(code, alpha)
    _check("trsm_llnn_noalloc", fn(code, m, n, al, _ptr(A), lda, _ptr(B), ldb, _stream(stream)))


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
ERR_DEVICE_TIMEOUT = 901


def trsm_device_status(clear: bool = True) -> int:
    """Device-side status (0, or 901 when a kernel's bounded wait expired);
    synchronises the current device."""
    fn = load_library().trsm_device_status
    fn.argtypes = [ctypes.c_int]
    fn.restype = ctypes.c_int
    return int(fn(1 if clear else 0))


def trsm_set_wait_limit(polls: int) -> None:
    """Testing hook: polls of the batched f32 small kernel's first wait per
    item (0: expire at once; negative: the compiled limit).  See
    include/trsm.h."""
    fn = load_library().trsm_set_wait_limit
    fn.argtypes = [ctypes.c_int64]
    fn.restype = ctypes.c_int
    _check("trsm_set_wait_limit", fn(int(polls)))


def trsm_status_string(status: int) -> str:
    return load_library().trsm_status_string(int(status)).decode()


# ------------------------------------------------------------------ convenience
def solve(A, B, alpha=1.0, stream=None):
    """Solve L X = alpha B in place in ``B`` for CUDA tensors.

    ``A`` is (m, m) or (batch, m, m), ``B`` is (m, n) or (batch, m, n), both
    of one of float32 / float64 / complex64 / complex128.  Each matrix must be
    column-major (stride (1, ld)) or row-major (stride (ld, 1)), both in the
    same layout; the batch dimension may have any stride.  Returns ``B``.
    """
    import torch
    if A.dtype != B.dtype:
        raise TypeError("A and B must have the same dtype")
    batched = B.dim() == 3
    if A.dim() != B.dim() or B.dim() not in (2, 3):
        raise ValueError("expected A (m, m) / B (m, n), or batched (batch, m, m) / (batch, m, n)")
    m, n = B.shape[-2], B.shape[-1]
    if A.shape[-2:] != (m, m):
        raise ValueError("A must be square with as many rows as B")

    def geom(t, rows, cols):
        s0, s1 = t.stride(-2), t.stride(-1)
        if s0 == 1 and (s1 >= max(1, rows) or cols <= 1):
            return "col", max(s1, rows, 1)
        if s1 == 1 and (s0 >= max(1, cols) or rows <= 1):
            return "row", max(s0, cols, 1)
        raise ValueError("each matrix must be column-major or row-major (unit stride in one dim)")

    la, lda = geom(A, m, m)
    lb, ldb = geom(B, m, n)
    if la != lb:
        if m <= 1:
            la = lb
        else:
            raise ValueError("A and B must share one layout")
    code = _dtype_code(B.dtype)
    batch = B.shape[0] if batched else 1
    sa = A.stride(0) if batched else 0
    sb = B.stride(0) if batched else 0
    trsm_llnn_strided_batched(code, lb, m, n, alpha, A, lda, sa, B, ldb, sb, batch, stream)
    return B
