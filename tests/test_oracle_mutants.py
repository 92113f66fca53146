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
