"""The C-ABI library builds, loads and exports every symbol include/trsm.h
declares; host-only entry points and argument checking work without a GPU
(no call here reaches a kernel launch)."""
import ctypes

import pytest

import triangular_solve_gb300 as tg


@pytest.fixture(scope="module")
def lib():
    from triangular_solve_gb300 import build
    build.build()
    return tg.load_library()


EXPECTED = {"trsm_llnn", "trsm_llnn_strided_batched", "trsm_llnn_strided_batched_host", "trsm_llnn_select_nb",
            "trsm_llnn_workspace_bytes", "trsm_llnn_ex", "trsm_llnn_profile", "trsm_trtri_lower",
            "trsm_general", "trsm_status_string"}


def test_header_declares_the_boundary():
    assert EXPECTED <= set(tg.declared_functions())


def test_every_declared_symbol_is_exported(lib):
    for name in tg.declared_functions():
        assert hasattr(lib, name), name


def test_no_torch_types_in_the_header():
    text = open(tg.HEADER).read()
    assert "torch" not in text.lower().replace("torch.complex", "")
    assert "extern \"C\"" in text


def test_select_nb_table(lib):
    assert tg.trsm_llnn_select_nb("f64", 64, 64) == 0
    for d in tg.DTYPES:
        for m in (65, 1000, 1024, 3000, 16384, 100000):
            assert tg.trsm_llnn_select_nb(d, m, m) in (128, 256, 512)
    with pytest.raises(tg.TrsmError):
        tg.trsm_llnn_select_nb(9, 100, 100)


def test_workspace_bytes(lib):
    assert tg.trsm_llnn_workspace_bytes("f32", 64, 64) == 0
    assert tg.trsm_llnn_workspace_bytes("f32", 1000, 0) == 0
    # m = 1000, NB = 128: 8 blocks of 128 x 128 plus two 128 x 72 panels (row
    # length rounded up to 4 elements), 4 bytes
    w = 8 * 128 * 128 * 4
    x = 128 * 72 * 4
    r = lambda v: (v + 255) // 256 * 256  # noqa: E731
    # f32 also holds the TF32 head/tail copies of the tensor-core operands:
    # the A panel (m x NB), the X panel (n x NB) and the split X_t the apply
    # leaves for the update (n x NB)
    tc = 2 * r(1000 * 128 * 4) + 4 * r(70 * 128 * 4)
    assert tg.trsm_llnn_workspace_bytes("f32", 1000, 70, 128) == r(w) + 2 * r(x) + tc
    assert tg.trsm_llnn_workspace_bytes("c128", 1000, 70, 512) == r(2 * 512 * 512 * 16) + 2 * r(512 * 72 * 16)
    with pytest.raises(ValueError):
        tg.trsm_llnn_workspace_bytes("f32", 1000, 70, 100)


def test_workspace_bytes_few_rhs(lib):
    """n <= 8: at least the few-right-hand-side kernel's data -- the inverted
    128-row diagonal blocks and the published copy of X (ceil(m/128) block
    rows of 128 x n), each rounded up to 256 bytes."""
    r = lambda v: (v + 255) // 256 * 256  # noqa: E731
    for d, e in (("f64", 8), ("c128", 16)):
        for m, n in ((4096, 1), (16384, 8), (1000, 3)):
            tb = (m + 127) // 128
            few = r(tb * 128 * 128 * e) + r(tb * n * 128 * e)
            for nb in (128, 256, 512):
                tbn = (m + nb - 1) // nb
                blocked = r(tbn * nb * nb * e) + 2 * r(nb * ((n + 3) // 4 * 4) * e)
                assert tg.trsm_llnn_workspace_bytes(d, m, n, nb) == max(few, blocked)
    # from nine columns on only the blocked path's own terms
    assert tg.trsm_llnn_workspace_bytes("f64", 4096, 9, 128) == r(32 * 128 * 128 * 8) + 2 * r(128 * 12 * 8)


def test_workspace_bytes_lookahead_form(lib):
    """f32 with n >= 256 and a last block of at least 16 rows takes the
    look-ahead form; its panels (rows padded to 256): the scaled L panel and
    the L panel twice each (m rows), the split block row three times (n
    rows), six NB x NB blocks -- head and tail each."""
    r = lambda v: (v + 255) // 256 * 256  # noqa: E731
    m, n, nb = 1000, 777, 256
    base = r(4 * nb * nb * 4) + 2 * r(nb * 780 * 4)
    per_block = 2 * r(m * nb * 4) + 4 * r(n * nb * 4)
    fused = 8 * r(1024 * nb * 4) + 6 * r(1024 * nb * 4) + 6 * r(nb * nb * 4)
    assert tg.trsm_llnn_workspace_bytes("f32", m, n, nb) == base + max(per_block, fused)
    # c64 in real form: W' (m rows) twice, the L panel's X' (2m rows) once,
    # R_t's X' (2n rows) three times, four NB x 2NB blocks; 2 NB floats a row
    base64 = r(4 * nb * nb * 8) + 2 * r(nb * 780 * 8)
    per_block64 = 2 * r(m * 2 * nb * 4) + 4 * r(2 * n * 2 * nb * 4)
    fused64 = 4 * r(1024 * 2 * nb * 4) + 2 * r(2048 * 2 * nb * 4) + 6 * r(2048 * 2 * nb * 4) + \
        4 * r(nb * 2 * nb * 4)
    assert tg.trsm_llnn_workspace_bytes("c64", m, n, nb) == base64 + max(per_block64, fused64)
    # an 8-row last block keeps the per-block flow
    assert tg.trsm_llnn_workspace_bytes("f32", 520, 300, 256) == \
        r(3 * nb * nb * 4) + 2 * r(nb * 300 * 4) + 2 * r(520 * nb * 4) + 4 * r(300 * nb * 4)


def test_lookahead_gates_at_their_boundaries(lib):
    """The look-ahead forms' gates, seen through the workspace they need:
    f32 from n = 256 columns; c64 from n = 256 up to n = 8192 (above that the
    per-block flow stays, measured faster once the split block row exceeds
    twice the L2)."""
    r = lambda v: (v + 255) // 256 * 256  # noqa: E731
    m, nb = 1000, 256
    rows = 1024  # m rounded up to 256

    def base(n, eb):
        return r(4 * nb * nb * eb) + 2 * r(nb * ((n + 3) // 4 * 4) * eb)

    def f32_per_block(n):
        return 2 * r(m * nb * 4) + 4 * r(n * nb * 4)

    def f32_fused(n):
        return 8 * r(rows * nb * 4) + 6 * r(r(n) * nb * 4) + 6 * r(nb * nb * 4)

    assert tg.trsm_llnn_workspace_bytes("f32", m, 255, nb) == base(255, 4) + f32_per_block(255)
    assert tg.trsm_llnn_workspace_bytes("f32", m, 256, nb) == base(256, 4) + max(f32_per_block(256), f32_fused(256))

    def c64_per_block(mm, n, b):
        return 2 * r(mm * 2 * b * 4) + 4 * r(2 * n * 2 * b * 4)

    def c64_fused(mm, n, b):
        ra, rx = r(mm), r(n)
        return 4 * r(ra * 2 * b * 4) + 2 * r(2 * ra * 2 * b * 4) + 6 * r(2 * rx * 2 * b * 4) + 4 * r(b * 2 * b * 4)

    mm, b = 16384, 512
    tbk = mm // b

    def base64(n):
        return r(tbk * b * b * 8) + 2 * r(b * ((n + 3) // 4 * 4) * 8)

    assert tg.trsm_llnn_workspace_bytes("c64", mm, 8192, b) == \
        base64(8192) + max(c64_per_block(mm, 8192, b), c64_fused(mm, 8192, b))
    assert tg.trsm_llnn_workspace_bytes("c64", mm, 8193, b) == base64(8193) + c64_per_block(mm, 8193, b)


def test_status_strings(lib):
    assert tg.trsm_status_string(0) == "success"
    assert "invalid argument" in tg.trsm_status_string(-3)
    assert "workspace" in tg.trsm_status_string(tg.ERR_WORKSPACE)


def _call(lib, *args):
    return lib.trsm_llnn(*args)


def test_argument_errors_report_position(lib):
    one = ctypes.byref(ctypes.c_double(1.0))
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    assert lib.trsm_llnn(7, 4, 4, one, fake, 4, fake, 4, None) == -1
    assert lib.trsm_llnn(1, -1, 4, one, fake, 4, fake, 4, None) == -2
    assert lib.trsm_llnn(1, 4, -1, one, fake, 4, fake, 4, None) == -3
    assert lib.trsm_llnn(1, 4, 4, None, fake, 4, fake, 4, None) == -4
    assert lib.trsm_llnn(1, 4, 4, one, None, 4, fake, 4, None) == -5
    assert lib.trsm_llnn(1, 4, 4, one, fake, 3, fake, 4, None) == -6
    assert lib.trsm_llnn(1, 4, 4, one, fake, 4, None, 4, None) == -7
    assert lib.trsm_llnn(1, 4, 4, one, fake, 4, fake, 3, None) == -8
    assert lib.trsm_llnn(1, 4, 4, one, fake + 4, 4, fake, 4, None) == -5  # misaligned double
    # quick returns touch nothing
    assert lib.trsm_llnn(1, 0, 4, one, None, 1, None, 1, None) == 0
    assert lib.trsm_llnn(1, 4, 0, one, None, 4, None, 4, None) == 0


def test_batched_argument_errors(lib):
    one = ctypes.byref(ctypes.c_float(1.0))
    fake = 1 << 20
    f = lib.trsm_llnn_strided_batched
    assert f(0, 2, 4, 4, one, fake, 4, 16, fake, 4, 16, 2, None) == -2
    assert f(0, 0, 4, 4, one, fake, 4, -1, fake, 4, 16, 2, None) == -8
    assert f(0, 1, 4, 6, one, fake, 4, 16, fake, 5, 30, 2, None) == -10   # row-major ldb < n
    assert f(0, 0, 4, 4, one, fake, 4, 16, fake, 4, 15, 2, None) == -11   # overlapping B
    assert f(0, 0, 4, 4, one, fake, 4, 16, fake, 4, 16, -1, None) == -12
    assert f(0, 0, 4, 4, one, fake, 4, 16, fake, 4, 16, 0, None) == 0


def test_ex_rejects_bad_block_size_and_workspace(lib):
    one = ctypes.byref(ctypes.c_double(1.0))
    fake = 1 << 20
    assert lib.trsm_llnn_ex(1, 200, 4, one, fake, 200, fake, 200, 100, fake, 1 << 30, None) == -9
    assert lib.trsm_llnn_ex(1, 200, 4, one, fake, 200, fake, 200, 128, None, 0, None) == tg.ERR_WORKSPACE
    assert lib.trsm_llnn_ex(1, 200, 4, one, fake, 200, fake, 200, 128, fake + 8, 1 << 30, None) == \
        tg.ERR_WORKSPACE
    assert lib.trsm_llnn_ex(1, 200, 4, one, fake, 200, fake, 200, 128, fake, 16, None) == tg.ERR_WORKSPACE


def test_cpu_tensors_are_refused():
    torch = pytest.importorskip("torch")
    A = torch.eye(4, dtype=torch.float64)
    B = torch.ones(4, 2, dtype=torch.float64)
    with pytest.raises(ValueError):
        tg.solve(A, B)


def test_host_entry_argument_errors_and_quick_returns(lib):
    """trsm_llnn_strided_batched_host validates like the device entry point
    and returns before touching any memory or device on quick returns."""
    one = ctypes.byref(ctypes.c_float(1.0))
    fake = 1 << 20  # never dereferenced
    f = lib.trsm_llnn_strided_batched_host
    assert f(9, 0, 4, 4, one, fake, 4, 16, fake, 4, 16, 2, None) == -1
    assert f(0, 2, 4, 4, one, fake, 4, 16, fake, 4, 16, 2, None) == -2
    assert f(0, 0, -1, 4, one, fake, 4, 16, fake, 4, 16, 2, None) == -3
    assert f(0, 0, 4, -1, one, fake, 4, 16, fake, 4, 16, 2, None) == -4
    assert f(0, 0, 4, 4, None, fake, 4, 16, fake, 4, 16, 2, None) == -5
    assert f(0, 0, 4, 4, one, None, 4, 16, fake, 4, 16, 2, None) == -6
    assert f(0, 0, 4, 4, one, fake, 3, 16, fake, 4, 16, 2, None) == -7
    assert f(0, 0, 4, 4, one, fake, 4, -1, fake, 4, 16, 2, None) == -8
    assert f(0, 0, 4, 4, one, fake, 4, 16, None, 4, 16, 2, None) == -9
    assert f(0, 0, 4, 4, one, fake, 4, 16, fake, 3, 16, 2, None) == -10
    assert f(0, 0, 4, 4, one, fake, 4, 16, fake, 4, 15, 2, None) == -11
    assert f(0, 0, 4, 4, one, fake, 4, 16, fake, 4, 16, -1, None) == -12
    assert f(0, 0, 0, 4, one, None, 1, 0, None, 1, 4, 2, None) == 0
    assert f(0, 0, 4, 0, one, None, 4, 0, None, 4, 0, 2, None) == 0
    assert f(0, 0, 4, 4, one, None, 4, 16, None, 4, 16, 0, None) == 0


def test_trtri_argument_errors_and_quick_return(lib):
    fake = 1 << 20  # never dereferenced: every call below fails validation first
    f = lib.trsm_trtri_lower
    assert f(9, 4, fake, 4, fake, 4, None) == -1
    assert f(0, -1, fake, 4, fake, 4, None) == -2
    assert f(0, 4, None, 4, fake, 4, None) == -3
    assert f(1, 4, fake + 4, 4, fake, 4, None) == -3   # misaligned double
    assert f(0, 4, fake, 3, fake, 4, None) == -4
    assert f(0, 4, fake, 4, None, 4, None) == -5
    assert f(0, 4, fake, 4, fake, 3, None) == -6
    assert f(0, 0, None, 1, None, 1, None) == 0


def test_general_variant_argument_errors_and_quick_returns(lib):
    one = ctypes.byref(ctypes.c_double(1.0))
    fake = 1 << 20  # never dereferenced: every call below fails validation or returns first
    f = lib.trsm_general
    assert f(7, 0, 0, 0, 0, 4, 4, one, fake, 4, fake, 4, None) == -1
    assert f(1, 2, 0, 0, 0, 4, 4, one, fake, 4, fake, 4, None) == -2
    assert f(1, 0, 2, 0, 0, 4, 4, one, fake, 4, fake, 4, None) == -3
    assert f(1, 0, 0, 3, 0, 4, 4, one, fake, 4, fake, 4, None) == -4
    assert f(1, 0, 0, 0, 2, 4, 4, one, fake, 4, fake, 4, None) == -5
    assert f(1, 0, 0, 0, 0, -1, 4, one, fake, 4, fake, 4, None) == -6
    assert f(1, 0, 0, 0, 0, 4, -1, one, fake, 4, fake, 4, None) == -7
    assert f(1, 0, 0, 0, 0, 4, 4, None, fake, 4, fake, 4, None) == -8
    assert f(1, 1, 1, 1, 1, 4, 6, one, None, 6, fake, 4, None) == -9
    assert f(1, 1, 0, 0, 0, 4, 6, one, fake, 5, fake, 4, None) == -10   # right side: lda >= n
    assert f(1, 0, 1, 0, 0, 4, 6, one, fake, 4, None, 4, None) == -11
    assert f(1, 0, 1, 0, 0, 4, 6, one, fake, 4, fake, 3, None) == -12
    assert f(1, 1, 1, 2, 1, 0, 6, one, None, 6, None, 1, None) == 0
    assert f(1, 1, 1, 2, 1, 4, 0, one, None, 1, None, 4, None) == 0


def test_general_variant_flags_in_the_binding():
    """side / uplo / trans / diag accept the BLAS letters (either case) or the
    header's enum values, and refuse anything else before the library is
    called."""
    assert tg._flag(tg._SIDE, "r", "side") == 1 and tg._flag(tg._SIDE, 0, "side") == 0
    assert tg._flag(tg._UPLO, "U", "uplo") == 1
    assert tg._flag(tg._OP, "c", "trans") == 2 and tg._flag(tg._OP, "T", "trans") == 1
    assert tg._flag(tg._DIAG, "u", "diag") == 1
    for table, bad in ((tg._SIDE, "X"), (tg._UPLO, 2), (tg._OP, "H"), (tg._DIAG, None)):
        with pytest.raises(ValueError):
            tg._flag(table, bad, "flag")
    with pytest.raises(ValueError):
        tg.trsm_general("f32", "Q", "L", "N", "N", 4, 4, 1.0, None, 4, None, 4)


def test_small_regime_rejects_too_many_columns(lib):
    one = ctypes.byref(ctypes.c_double(1.0))
    fake = 1 << 20
    n = 64 * 65535 + 1  # beyond the small kernels' column grid
    assert lib.trsm_llnn(1, 64, n, one, fake, 64, fake, 64, None) == -3
