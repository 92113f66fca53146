"""Planted mistakes in the oracle must turn its pins red (CPU only).

Each mutant is a copy of the oracle's C source with one plausible mistake (a
dropped term, a wrong sign, a transposed operand, an off-by-one info, a pivot
test that lets zero or NaN through). It is compiled into a temporary library
and run through a battery built from the same pins as test_oracle.py; every
mutant must fail at least one of them, and the unmutated source must pass all.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import pytest

import synth
from tests import checks
from tests.test_oracle import _brute, _integer_factor

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "chol_ref.c")

MUTANTS = {
    "identity": ("", ""),
    "pivot sign": ("d -= ljk * ljk;", "d += ljk * ljk;"),
    "dropped pivot term": ("for (int k = 0; k < j; ++k) {", "for (int k = 1; k < j; ++k) {"),
    "dropped update term": ("for (int k = 0; k < j; ++k)\n                s -=",
                            "for (int k = 0; k + 1 < j; ++k)\n                s -="),
    "transposed operand": ("s -= L[i + (int64_t)k * ldl] * L[j + (int64_t)k * ldl];",
                           "s -= L[i + (int64_t)k * ldl] * L[k + (int64_t)j * ldl];"),
    "multiply instead of divide": ("L[i + (int64_t)j * ldl] = s / ljj;",
                                   "L[i + (int64_t)j * ldl] = s * ljj;"),
    "info zero-based": ("return j + 1;", "return j;"),
    "zero pivot passes": ("if (!(d > 0.0))", "if (d < 0.0)"),
    "nan pivot passes": ("if (!(d > 0.0))", "if (d <= 0.0)"),
    "upper triangle read": ("double s = (double)A[i + (int64_t)j * lda];",
                            "double s = (double)A[j + (int64_t)i * lda];"),
}


def _compile(name: str, tmp_path) -> ctypes.CDLL:
    old, new = MUTANTS[name]
    src = open(SRC).read()
    if old:
        assert old in src, f"mutation site for {name!r} not found"
        src = src.replace(old, new, 1)
    c = tmp_path / "m.c"
    so = tmp_path / "m.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(c), "-o", str(so), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    lib.oracle_potrf_one.restype = ctypes.c_int
    lib.oracle_potrf_one.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_void_p, ctypes.c_int]
    return lib


def _potrf(lib, A):
    a32 = np.asfortranarray(np.asarray(A, dtype=np.float32))
    n = a32.shape[0]
    L = np.zeros((n, n), order="F")
    info = lib.oracle_potrf_one(a32.ctypes.data, n, n, L.ctypes.data, n)
    return np.ascontiguousarray(L), info


def _battery(lib) -> list[str]:
    """Names of the pins that fail for this library."""
    failed = []
    # exact integer factor, with a poisoned upper triangle
    L = _integer_factor(16, 16)
    A = (L @ L.T).astype(np.float32)
    Ap = np.tril(A) + np.triu(np.full_like(A, 1e30), 1)
    Lo, info = _potrf(lib, Ap)
    if info != 0 or not np.array_equal(Lo, L.astype(np.float64)):
        failed.append("integer factor")
    # brute force n = 3, 4
    g = np.random.default_rng(11)
    for n in (3, 4):
        for t in range(20):
            G = g.standard_normal((n, n))
            A = (G @ G.T + 0.1 * np.eye(n)) if t % 2 else (G + G.T)
            A32 = A.astype(np.float32)
            Lb, ib = _brute(A32)
            Lo, io = _potrf(lib, A32)
            m = n if ib == 0 else ib - 1
            if io != ib or (m and not np.allclose(Lo[:, :m], Lb[:, :m], rtol=1e-9, atol=1e-12)):
                failed.append(f"brute n={n}")
                break
    # diagonal with a zero and a NaN pivot
    for v in (0.0, np.nan):
        d = np.array([1.0, 4.0, v, 9.0], dtype=np.float32)
        if _potrf(lib, np.diag(d))[1] != 3:
            failed.append(f"diagonal {v}")
    # indefinite by construction, failing pivot behind a positive diagonal
    w = synth.WORKLOADS["n64"]
    for k in (0, 20, 63):
        A32 = synth.make_indefinite(synth.spd_matrix(w, k), k, delta=0.05).astype(np.float32)
        if _potrf(lib, A32)[1] != k + 1:
            failed.append(f"info k={k}")
            break
    # reconstruction budget on a workload matrix
    A32 = synth.spd_matrix(w, 2).astype(np.float32)
    Lo, info = _potrf(lib, A32)
    if info != 0 or not checks.recon_error(Lo, np.tril(A32)) <= 1e-13:
        failed.append("reconstruction")
    return failed


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    failed = _battery(_compile(name, tmp_path))
    if name == "identity":
        assert failed == [], failed
    else:
        assert failed, f"planted mistake {name!r} passed every pin"


# --------------------------------------------------------------------------
# The SPOTRS oracle (forward and backward substitution with the factor)
# --------------------------------------------------------------------------

SRC_TRS = os.path.join(os.path.dirname(SRC), "potrs_ref.c")

TRS_MUTANTS = {
    "identity": ("", ""),
    "forward reads the upper triangle": ("s -= (double)L[i + (int64_t)k * lda] * x[k];",
                                         "s -= (double)L[k + (int64_t)i * lda] * x[k];"),
    "backward not transposed": ("s -= (double)L[k + (int64_t)i * lda] * x[k];",
                                "s -= (double)L[i + (int64_t)k * lda] * x[k];"),
    "backward skipped": ("for (int i = n - 1; i >= 0; --i) {", "for (int i = n - 1; i >= n; --i) {"),
    "dropped forward term": ("for (int k = 0; k < i; ++k)", "for (int k = 1; k < i; ++k)"),
    "dropped backward term": ("for (int k = i + 1; k < n; ++k)", "for (int k = i + 2; k < n; ++k)"),
    "multiply instead of divide": ("x[i] = s / (double)L[i + (int64_t)i * lda];",
                                   "x[i] = s * (double)L[i + (int64_t)i * lda];"),
}


def _compile_trs(name: str, tmp_path) -> ctypes.CDLL:
    old, new = TRS_MUTANTS[name]
    src = open(SRC_TRS).read()
    if old:
        assert old in src, f"mutation site for {name!r} not found"
        src = src.replace(old, new, 1)
    c = tmp_path / "t.c"
    so = tmp_path / "t.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(c), "-o", str(so), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    lib.oracle_potrs_one.restype = None
    lib.oracle_potrs_one.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
    return lib


def _potrs(lib, L, B):
    l32 = np.asfortranarray(np.asarray(L, dtype=np.float32))
    b32 = np.asfortranarray(np.asarray(B, dtype=np.float32))
    n, nrhs = b32.shape
    X = np.zeros((n, nrhs), order="F")
    lib.oracle_potrs_one(l32.ctypes.data, n, n, b32.ctypes.data, nrhs, n, X.ctypes.data, n)
    return np.ascontiguousarray(X)


def _trs_battery(lib) -> list[str]:
    from tests.test_oracle_potrs import _int_factor
    failed = []
    # exact integer solution with a poisoned upper triangle
    n = 9
    L = _int_factor(n, 3)
    X = np.random.default_rng(4).integers(-5, 6, (n, 3)).astype(np.float64)
    B = L @ (L.T @ X)
    Lp = L + np.triu(np.full((n, n), 1e30), 1)
    if not np.array_equal(_potrs(lib, Lp, B), X):
        failed.append("integer solution")
    # backward error on a well-conditioned factor
    g = np.random.default_rng(6)
    G = g.standard_normal((40, 40))
    Lw = np.linalg.cholesky(G @ G.T / 40 + np.eye(40)).astype(np.float32).astype(np.float64)
    Bw = g.standard_normal((40, 2)).astype(np.float32).astype(np.float64)
    Xw = _potrs(lib, Lw, Bw)
    r = np.linalg.norm(Lw @ (Lw.T @ Xw) - Bw)
    if not (r <= 10 * 40 * 2.0 ** -53 * np.linalg.norm(Lw) ** 2 * np.linalg.norm(Xw)):
        failed.append("backward error")
    return failed


@pytest.mark.parametrize("name", list(TRS_MUTANTS))
def test_trs_mutant_is_caught(name, tmp_path):
    failed = _trs_battery(_compile_trs(name, tmp_path))
    if name == "identity":
        assert failed == [], failed
    else:
        assert failed, f"planted mistake {name!r} passed every pin"


# --------------------------------------------------------------------------
# uplo = 'U': mistakes planted in the upper-triangle functions only
# --------------------------------------------------------------------------

UPPER_MUTANTS = {
    "identity": ("", ""),
    "pivot sign": ("d -= ukj * ukj;", "d += ukj * ukj;"),
    "lower triangle read": ("double s = (double)A[j + (int64_t)i * lda];",
                            "double s = (double)A[i + (int64_t)j * lda];"),
    "transposed operand": ("s -= U[k + (int64_t)j * ldu] * U[k + (int64_t)i * ldu];",
                           "s -= U[k + (int64_t)j * ldu] * U[i + (int64_t)k * ldu];"),
    "dropped update term": ("for (int k = 0; k < j; ++k)\n                s -=",
                            "for (int k = 0; k + 1 < j; ++k)\n                s -="),
    "info zero-based": ("return j + 1;", "return j;"),
    "zero pivot passes": ("if (!(d > 0.0))", "if (d < 0.0)"),
}

UPPER_TRS_MUTANTS = {
    "identity": ("", ""),
    "forward reads the lower triangle": ("s -= (double)U[k + (int64_t)i * lda] * x[k];",
                                         "s -= (double)U[i + (int64_t)k * lda] * x[k];"),
    "backward transposed": ("s -= (double)U[i + (int64_t)k * lda] * x[k];",
                            "s -= (double)U[k + (int64_t)i * lda] * x[k];"),
    "backward skipped": ("for (int i = n - 1; i >= 0; --i) {", "for (int i = n - 1; i >= n; --i) {"),
    "dropped forward term": ("for (int k = 0; k < i; ++k)", "for (int k = 1; k < i; ++k)"),
}


def _compile_after(src_path: str, marker: str, old: str, new: str, tmp_path, tag: str):
    """Compile ``src_path`` with the first ``old`` after ``marker`` replaced."""
    src = open(src_path).read()
    if old:
        at = src.index(marker)
        pos = src.index(old, at)
        src = src[:pos] + new + src[pos + len(old):]
    c = tmp_path / f"{tag}.c"
    so = tmp_path / f"{tag}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(c), "-o", str(so), "-lm"], check=True)
    return ctypes.CDLL(str(so))


def _potrf_upper(lib, A):
    a32 = np.asfortranarray(np.asarray(A, dtype=np.float32))
    n = a32.shape[0]
    U = np.zeros((n, n), order="F")
    info = lib.oracle_potrf_upper_one(a32.ctypes.data, n, n, U.ctypes.data, n)
    return np.ascontiguousarray(U), info


def _upper_battery(lib) -> list[str]:
    from tests.test_oracle_upper import _int_upper
    lib.oracle_potrf_upper_one.restype = ctypes.c_int
    lib.oracle_potrf_upper_one.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_int]
    failed = []
    U = _int_upper(16, 17)
    A = (U.T @ U).astype(np.float32)
    Ap = np.triu(A) + np.tril(np.full_like(A, 1e30), -1)
    Uo, info = _potrf_upper(lib, Ap)
    if info != 0 or not np.array_equal(Uo, U):
        failed.append("integer factor")
    g = np.random.default_rng(12)
    for n in (3, 4):
        for t in range(20):
            G = g.standard_normal((n, n))
            A32 = ((G @ G.T + 0.1 * np.eye(n)) if t % 2 else (G + G.T)).astype(np.float32)
            Lb, ib = _brute(np.ascontiguousarray(A32.T))
            Uo, io = _potrf_upper(lib, A32)
            m = n if ib == 0 else ib - 1
            if io != ib or (m and not np.allclose(Uo[:m, :], Lb[:, :m].T, rtol=1e-9,
                                                  atol=1e-12)):
                failed.append(f"brute n={n}")
                break
    d = np.array([1.0, 4.0, 0.0, 9.0], dtype=np.float32)
    if _potrf_upper(lib, np.diag(d))[1] != 3:
        failed.append("diagonal zero")
    return failed


@pytest.mark.parametrize("name", list(UPPER_MUTANTS))
def test_upper_mutant_is_caught(name, tmp_path):
    old, new = UPPER_MUTANTS[name]
    lib = _compile_after(SRC, "int oracle_potrf_upper_one(", old, new, tmp_path, "u")
    failed = _upper_battery(lib)
    if name == "identity":
        assert failed == [], failed
    else:
        assert failed, f"planted mistake {name!r} passed every pin"


def _upper_trs_battery(lib) -> list[str]:
    from tests.test_oracle_upper import _int_upper
    lib.oracle_potrs_upper_one.restype = None
    lib.oracle_potrs_upper_one.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_int]
    failed = []
    n = 9
    U = _int_upper(n, 5)
    X = np.random.default_rng(6).integers(-5, 6, (n, 3)).astype(np.float64)
    B = U.T @ (U @ X)
    Up = np.asfortranarray((U + np.tril(np.full((n, n), 1e30), -1)).astype(np.float32))
    b32 = np.asfortranarray(B.astype(np.float32))
    Xo = np.zeros((n, 3), order="F")
    lib.oracle_potrs_upper_one(Up.ctypes.data, n, n, b32.ctypes.data, 3, n, Xo.ctypes.data, n)
    if not np.array_equal(Xo, X):
        failed.append("integer solution")
    return failed


@pytest.mark.parametrize("name", list(UPPER_TRS_MUTANTS))
def test_upper_trs_mutant_is_caught(name, tmp_path):
    old, new = UPPER_TRS_MUTANTS[name]
    lib = _compile_after(SRC_TRS, "void oracle_potrs_upper_one(", old, new, tmp_path, "ut")
    failed = _upper_trs_battery(lib)
    if name == "identity":
        assert failed == [], failed
    else:
        assert failed, f"planted mistake {name!r} passed every pin"
