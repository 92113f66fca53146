"""The C-ABI library builds, loads and exports what include/*.h declares; the
host-side logic (argument checks, quick returns, route selection) works without
a GPU; every kernel compiles with no stack frame and no spills (CPU only)."""
from __future__ import annotations

import glob
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(
    shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
    reason="nvcc not available")


@pytest.fixture(scope="module")
def bl():
    from matrix_dense_linear_gb300 import build
    build.build()
    import matrix_dense_linear_gb300 as bl
    bl.library()
    return bl


def _declared_functions() -> set[str]:
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(bl_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(bl):
    declared = _declared_functions()
    assert "bl_spotrf_batched" in declared and "bl_spotrf_batched_ex" in declared
    lib = bl.library()
    for name in declared:
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert declared == set(bl.SYMBOLS), "binding and header disagree"


def test_version(bl):
    assert bl.version().startswith("bl_spotrf ") and "sm_103a" in bl.version()


@pytest.mark.parametrize("args,code", [
    # (A, n, lda, strideA, batch, info) -> status; no call below reaches the GPU
    ((8, -1, 1, 1, 1, 8), -2),
    ((8, 4, 4, 16, -1, 8), -5),
    ((8, 4, 3, 16, 2, 8), -3),
    ((8, 0, 0, 0, 1, 8), -3),
    ((8, 4, 4, 15, 2, 8), -4),
    ((8, 4, 4, -16, 2, 8), -4),
    ((None, 4, 4, 16, 2, 8), -1),
    ((8, 4, 4, 16, 2, None), -6),
    ((8, 4097, 4097, 4097 * 4097, 2, 8), -7),
    ((None, 4, 4, 16, 0, None), 0),   # batch == 0: nothing to do
])
def test_argument_checks(bl, args, code):
    A, n, lda, sA, batch, info = args
    lib = bl.library()
    if code is None:
        return
    assert lib.bl_spotrf_batched(A, n, lda, sA, batch, info, None) == code
    assert lib.bl_spotrf_batched_ex(A, n, lda, sA, batch, info, None, 0) == code


def test_check_order(bl):
    lib = bl.library()
    # n < 0 wins over everything; then batch < 0; then lda
    assert lib.bl_spotrf_batched(None, -1, 0, 0, -1, None, None) == -2
    assert lib.bl_spotrf_batched(None, 4, 0, 0, -1, None, None) == -5
    assert lib.bl_spotrf_batched(None, 4, 1, 0, 2, None, None) == -3
    assert lib.bl_spotrf_batched(None, 4, 4, 1, 2, None, None) == -4


@pytest.mark.parametrize("args,code", [
    # (L, n, lda, strideA, B, nrhs, ldb, strideB, batch) -> status; nothing reaches the GPU
    ((8, -1, 1, 1, 8, 1, 1, 1, 1), -2),
    ((8, 4097, 4097, 4097 * 4097, 8, 1, 4097, 4097, 1), -2),
    ((8, 4, 4, 16, 8, -1, 4, 4, 1), -6),
    ((8, 4, 4, 16, 8, 2, 4, 8, -1), -9),
    ((8, 4, 3, 16, 8, 2, 4, 8, 2), -3),
    ((8, 4, 4, 16, 8, 2, 3, 8, 2), -7),
    ((8, 4, 4, 15, 8, 2, 4, 8, 2), -4),
    ((8, 4, 4, 16, 8, 2, 4, 7, 2), -8),
    ((None, 4, 4, 16, 8, 2, 4, 8, 2), -1),
    ((8, 4, 4, 16, None, 2, 4, 8, 2), -5),
    ((None, 4, 4, 16, None, 2, 4, 8, 0), 0),   # batch == 0: nothing to do
    ((None, 0, 1, 0, None, 2, 1, 2, 3), 0),    # n == 0
    ((None, 4, 4, 16, None, 0, 4, 0, 3), 0),   # nrhs == 0
])
def test_trs_argument_checks(bl, args, code):
    lib = bl.library()
    assert lib.bl_spotrs_batched(*args, None) == code
    L, n, lda, sA, B, nrhs, ldb, sB, batch = args
    if code != 0:
        assert lib.bl_sposv_batched(*args, 8, None) == code


def test_trs_check_order(bl):
    lib = bl.library()
    assert lib.bl_spotrs_batched(None, -1, 0, 0, None, -1, 0, 0, -1, None) == -2
    assert lib.bl_spotrs_batched(None, 4, 0, 0, None, -1, 0, 0, -1, None) == -6
    assert lib.bl_spotrs_batched(None, 4, 0, 0, None, 1, 0, 0, -1, None) == -9
    assert lib.bl_spotrs_batched(None, 4, 0, 0, None, 1, 0, 0, 2, None) == -3
    assert lib.bl_spotrs_batched(None, 4, 4, 0, None, 1, 0, 0, 2, None) == -7
    assert lib.bl_spotrs_batched(None, 4, 4, 0, None, 1, 4, 0, 2, None) == -4
    assert lib.bl_spotrs_batched(None, 4, 4, 16, None, 1, 4, 0, 2, None) == -8
    assert lib.bl_spotrs_batched(None, 4, 4, 16, None, 1, 4, 4, 2, None) == -1
    assert lib.bl_spotrs_batched(8, 4, 4, 16, None, 1, 4, 4, 2, None) == -5
    # sposv: info last
    assert lib.bl_sposv_batched(8, 4, 4, 16, 8, 1, 4, 4, 2, None, None) == -10
    assert lib.bl_sposv_batched(8, 4, 4, 16, None, 1, 4, 4, 2, None, None) == -5


@pytest.mark.parametrize("uplo", [b"U", b"u", b"L", b"l"])
def test_uplo_argument_codes_are_shifted(bl, uplo):
    """The uplo entry points take uplo as argument 1: every code of the call
    without it moves down by one (nothing below reaches the GPU)."""
    lib = bl.library()
    cases = [((8, -1, 1, 1, 1, 8), -2), ((8, 4, 4, 16, -1, 8), -5), ((8, 4, 3, 16, 2, 8), -3),
             ((8, 4, 4, 15, 2, 8), -4), ((None, 4, 4, 16, 2, 8), -1),
             ((8, 4, 4, 16, 2, None), -6), ((8, 4097, 4097, 4097 * 4097, 2, 8), -7)]
    for args, code in cases:
        assert lib.bl_spotrf_batched_uplo(uplo, *args, None) == code - 1
        assert lib.bl_spotrf_batched_uplo_ex(uplo, *args, None, 0) == code - 1
    assert lib.bl_spotrf_batched_uplo(uplo, None, 4, 4, 16, 0, None, None) == 0
    assert lib.bl_spotrf_batched_uplo_ex(uplo, 8, 65, 65, 65 * 65, 1, 8, None,
                                         bl.ROUTE_WARP) == -9
    assert lib.bl_spotrf_batched_uplo_ex(uplo, 8, 4, 4, 16, 1, 8, None, 9) == -9
    # solves: L/A -2, n -3, lda -4, strideA -5, B -6, nrhs -7, ldb -8, strideB -9, batch -10
    assert lib.bl_spotrs_batched_uplo(uplo, 8, -1, 1, 1, 8, 1, 1, 1, 1, None) == -3
    assert lib.bl_spotrs_batched_uplo(uplo, 8, 4, 4, 16, 8, 2, 4, 8, -1, None) == -10
    assert lib.bl_spotrs_batched_uplo(uplo, 8, 4, 4, 16, None, 2, 4, 8, 2, None) == -6
    assert lib.bl_sposv_batched_uplo(uplo, 8, 4, 4, 16, 8, 1, 4, 4, 2, None, None) == -11
    assert lib.bl_sposv_batched_uplo(uplo, None, 4, 4, 16, 8, 1, 4, 4, 2, 8, None) == -2


def test_bad_uplo(bl):
    lib = bl.library()
    for bad in (b"X", b"\x00", b"N"):
        assert lib.bl_spotrf_batched_uplo(bad, 8, 4, 4, 16, 1, 8, None) == -1
        assert lib.bl_spotrf_batched_uplo_ex(bad, 8, 4, 4, 16, 1, 8, None, 0) == -1
        assert lib.bl_spotrs_batched_uplo(bad, 8, 4, 4, 16, 8, 1, 4, 4, 1, None) == -1
        assert lib.bl_sposv_batched_uplo(bad, 8, 4, 4, 16, 8, 1, 4, 4, 1, 8, None) == -1


def test_dpotrf_argument_codes(bl):
    """The double call checks its arguments like the single one (nothing below
    reaches the GPU); its uplo form shifts them by one."""
    lib = bl.library()
    cases = [((8, -1, 1, 1, 1, 8), -2), ((8, 4, 4, 16, -1, 8), -5), ((8, 4, 3, 16, 2, 8), -3),
             ((8, 4, 4, 15, 2, 8), -4), ((None, 4, 4, 16, 2, 8), -1),
             ((8, 4, 4, 16, 2, None), -6), ((8, 4097, 4097, 4097 * 4097, 2, 8), -7)]
    for args, code in cases:
        assert lib.bl_dpotrf_batched(*args, None) == code
        assert lib.bl_dpotrf_batched_uplo(b"U", *args, None) == code - 1
    assert lib.bl_dpotrf_batched_uplo(b"Q", 8, 4, 4, 16, 1, 8, None) == -1
    assert lib.bl_dpotrf_batched(None, 4, 4, 16, 0, None, None) == 0


def test_cpotrf_argument_codes(bl):
    lib = bl.library()
    cases = [((8, -1, 1, 1, 1, 8), -2), ((8, 4, 4, 16, -1, 8), -5), ((8, 4, 3, 16, 2, 8), -3),
             ((8, 4, 4, 15, 2, 8), -4), ((None, 4, 4, 16, 2, 8), -1),
             ((8, 4, 4, 16, 2, None), -6), ((8, 4097, 4097, 4097 * 4097, 2, 8), -7),
             ((12, 4, 4, 16, 2, 8), -1)]  # not 8-byte aligned (the last case)
    for args, code in cases:
        assert lib.bl_cpotrf_batched(*args, None) == code
        assert lib.bl_cpotrf_batched_uplo(b"L", *args, None) == code - 1
    assert lib.bl_cpotrf_batched_uplo(b"?", 8, 4, 4, 16, 1, 8, None) == -1
    for args, code in cases[:-1]:
        assert lib.bl_zpotrf_batched(*args, None) == code
        assert lib.bl_zpotrf_batched_uplo(b"U", *args, None) == code - 1
    assert lib.bl_zpotrf_batched(8, 4, 4, 16, 2, 8, None) == -1  # not 16-byte aligned


def test_forced_route_that_cannot_run(bl):
    lib = bl.library()
    assert lib.bl_spotrf_batched_ex(8, 65, 65, 65 * 65, 1, 8, None, bl.ROUTE_WARP) == -8
    assert lib.bl_spotrf_batched_ex(8, 129, 129, 129 * 129, 1, 8, None, bl.ROUTE_CTA) == -8
    assert lib.bl_spotrf_batched_ex(8, 129, 129, 129 * 129, 1, 8, None, bl.ROUTE_TMEM) == -8
    assert lib.bl_spotrf_batched_ex(8, 4, 4, 16, 1, 8, None, bl.ROUTE_LEFT + 1) == -8
    assert lib.bl_spotrf_batched_ex(8, 128, 128, 128 * 128, 1, 8, None, bl.ROUTE_LEFT) == -8
    assert lib.bl_spotrf_batched_ex(8, 4, 4, 16, 1, 8, None, 9) == -8
    assert lib.bl_spotrf_batched_ex(8, 4, 4, 16, 1, 8, None, -1) == -8
    # argument errors come first
    assert lib.bl_spotrf_batched_ex(8, 65, 64, 65 * 65, 1, 8, None, bl.ROUTE_WARP) == -3


def test_route_selection(bl):
    assert bl.route(0, 5) == 0 and bl.route(5, 0) == 0
    for n in (1, 8, 9, 16, 17, 32, 33, 64):
        assert bl.route(n, 1024) == bl.ROUTE_WARP
    for n in (65, 100, 128):
        assert bl.route(n, 1024) == bl.ROUTE_CTA
    for n in (129, 256, 1024, 4096):
        assert bl.route(n, 8) == bl.ROUTE_BLOCKED
    # large batches above n = 256: the left-looking order (152 SMs assumed
    # without a device: batch x row tiles below the first panel >= 1520)
    assert bl.route(256, 4096) == bl.ROUTE_BLOCKED
    assert bl.route(1024, 512) == bl.ROUTE_LEFT
    assert bl.route(1024, 128) == bl.ROUTE_BLOCKED
    assert bl.route(2048, 128) == bl.ROUTE_LEFT


def test_no_stack_no_spill(bl):
    from matrix_dense_linear_gb300 import build
    rep = build.ptxas_report()
    funcs = re.findall(r"Function properties for (\S+)\n\s*(\d+) bytes stack frame, "
                       r"(\d+) bytes spill stores, (\d+) bytes spill loads", rep)
    assert len(funcs) >= 6, rep[:2000]
    for name, stack, st, ld in funcs:
        assert (int(stack), int(st), int(ld)) == (0, 0, 0), f"{name}: stack/spill {stack}/{st}/{ld}"


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import matrix_dense_linear_gb300 as bl
    monkeypatch.setattr(bl, "library_path", str(tmp_path / "absent.so"))
    monkeypatch.setattr(bl, "_lib", None)
    with pytest.raises(ImportError):
        bl.library()


def test_workspace_bytes(bl):
    """One 128 x 128 float block per matrix on the blocked route, none below it
    or for empty and out-of-range calls (host only)."""
    assert bl.workspace_bytes(128, 1000) == 0
    assert bl.workspace_bytes(129, 3) == 3 * 128 * 128 * 4
    assert bl.workspace_bytes(1024, 512) == 512 * 65536
    assert bl.workspace_bytes(4096, 1) == 65536
    assert bl.workspace_bytes(4097, 1) == 0
    assert bl.workspace_bytes(0, 5) == 0 and bl.workspace_bytes(512, 0) == 0
    assert bl.workspace_bytes(-3, 5) == 0 and bl.workspace_bytes(512, -1) == 0


def test_workspace_argument_codes(bl):
    """Checked on the host before anything is launched: the usual argument codes
    first, then -8 (work not 16-byte aligned) and -9 (too small); the uplo form
    counts uplo as argument 1."""
    lib = bl.library()
    need = bl.workspace_bytes(512, 2)
    assert lib.bl_spotrf_batched_ws(16, 512, 512, 512 * 512, 2, 16, 4100, need, None) == -8
    assert lib.bl_spotrf_batched_ws(16, 512, 512, 512 * 512, 2, 16, 4096, need - 4, None) == -9
    assert lib.bl_spotrf_batched_ws(16, 512, 511, 512 * 512, 2, 16, 4100, need, None) == -3
    assert lib.bl_spotrf_batched_ws(16, 512, 512, 512 * 512, 2, None, 4100, need, None) == -6
    assert lib.bl_spotrf_batched_uplo_ws(b"L", 16, 512, 512, 512 * 512, 2, 16, 4100, need,
                                         None) == -9
    assert lib.bl_spotrf_batched_uplo_ws(b"U", 16, 512, 512, 512 * 512, 2, 16, 4096, 0,
                                         None) == -10
    assert lib.bl_spotrf_batched_uplo_ws(b"Q", 16, 512, 512, 512 * 512, 2, 16, 4096, need,
                                         None) == -1


def test_host_call_argument_codes(bl):
    """bl_spotrf_batched_host checks its device buffers as A and info, then
    the host buffers (-1, -6), then the streams (-11), all before any copy."""
    import ctypes
    lib = bl.library()
    one = (ctypes.c_void_p * 1)(None)
    st = ctypes.addressof(one)
    # (A_host, n, lda, strideA, batch, info_host, A_dev, info_dev, streams, nstreams)
    cases = [
        ((16, 4, 4, 16, 2, 16, None, 16, st, 1), -1),
        ((16, 4, 4, 16, 2, 16, 16, None, st, 1), -6),
        ((16, 4, 3, 16, 2, 16, 16, 16, st, 1), -3),
        ((16, -1, 4, 16, 2, 16, 16, 16, st, 1), -2),
        ((16, 4, 4, 16, -1, 16, 16, 16, st, 1), -5),
        ((None, 4, 4, 16, 2, 16, 16, 16, st, 1), -1),
        ((16, 4, 4, 16, 2, None, 16, 16, st, 1), -6),
        ((16, 4, 4, 16, 2, 16, 16, 16, None, 1), -11),
        ((16, 4, 4, 16, 2, 16, 16, 16, st, 0), -11),
        ((None, 4, 4, 16, 0, None, None, None, st, 1), 0),  # batch == 0: nothing to do
    ]
    for (Ah, n, lda, sA, batch, ih, Ad, idv, streams, ns), code in cases:
        got = lib.bl_spotrf_batched_host(Ah, n, lda, sA, batch, ih, Ad, idv, 0, streams, ns)
        assert got == code, (n, lda, batch, got, code)


def test_static_call_scratch_limit(bl):
    """bl_spotrf_batched_static: the argument codes first, then -10 when the
    scratch the call would need passes the library's fixed array (checked on
    the host before anything is looked up or launched)."""
    lib = bl.library()
    per = bl.workspace_bytes(512, 1)
    fits = (16 << 20) // per  # matrices of order > 128 the 16 MB array holds
    assert fits == 256
    assert lib.bl_spotrf_batched_static(16, 512, 512, 512 * 512, fits + 1, 16, None) == -10
    assert lib.bl_spotrf_batched_static(16, 4096, 4096, 4096 * 4096, 1000, 16, None) == -10
    assert lib.bl_spotrf_batched_static(16, 512, 511, 512 * 512, fits + 1, 16, None) == -3
    assert lib.bl_spotrf_batched_static(16, 512, 512, 512 * 512, fits + 1, None, None) == -6
    assert lib.bl_spotrf_batched_static(None, 4, 4, 16, 0, None, None) == 0
