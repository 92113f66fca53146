"""Pins of the double-precision oracle (DPOTRF, lower and upper) against what
the mathematics fixes (CPU only): closed forms on inputs that are not float32
numbers, exact recovery of integer factors whose products need double
precision, leading minors in rational arithmetic, exact info, and bit-for-bit
agreement with the single-precision oracle (pinned on its own) wherever the
input is a float32 number. Planted mistakes must fail at least one pin.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
import synth
from tests import checks
from tests.test_oracle import _brute

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "dchol_ref.c")


def _int_lower(n: int, seed: int, big: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    L = np.tril(g.integers(-big, big + 1, (n, n)), -1).astype(np.float64)
    L[np.diag_indices(n)] = g.integers(1, big + 1, n)
    return L


@pytest.mark.parametrize("uplo", ["L", "U"])
def test_two_by_two_beyond_float(uplo):
    a, b, c = 2.0 + 2.0 ** -40, 1.0 + 2.0 ** -35, 3.0 - 2.0 ** -38
    assert float(np.float32(a)) != a  # not a float32 number
    L, info = oracle.dpotrf_one(np.array([[a, b], [b, c]]), uplo)
    assert info == 0
    l11 = math.sqrt(a)
    want = np.array([[l11, 0.0], [b / l11, math.sqrt(c - (b / l11) ** 2)]])
    np.testing.assert_allclose(L if uplo == "L" else L.T, want, rtol=1e-15)


@pytest.mark.parametrize("n", [2, 9, 40, 100])
@pytest.mark.parametrize("uplo", ["L", "U"])
def test_integer_factor_needing_double(n, uplo):
    # entries up to 2^13: A's entries pass 2^24 (not float32-exact) but stay
    # far below 2^53, so every intermediate is an exact double integer
    L = _int_lower(n, 30 + n, 2 ** 13)
    A = L @ L.T
    assert np.abs(A).max() > 2 ** 24 and np.abs(A).max() < 2 ** 50
    F, info = oracle.dpotrf_one(A, uplo)
    assert info == 0
    assert np.array_equal(F, L if uplo == "L" else L.T)


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_brute_force_small(n):
    g = np.random.default_rng(900 + n)
    for trial in range(30):
        if trial % 3 == 0:
            A = g.standard_normal((n, n))
            A = A + A.T
        else:
            G = g.standard_normal((n, n))
            A = G @ G.T + 0.05 * np.eye(n)
        A32 = A.astype(np.float32)  # _brute works on float32 inputs
        Lb, ib = _brute(A32)
        Lo, io = oracle.dpotrf_one(A32.astype(np.float64))
        assert io == ib
        m = n if ib == 0 else ib - 1
        if m:
            np.testing.assert_allclose(Lo[:, :m], Lb[:, :m], rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("name", ["n32", "n64", "n128"])
@pytest.mark.parametrize("uplo", ["L", "U"])
def test_equals_single_oracle_on_float_inputs(name, uplo):
    w = synth.WORKLOADS[name]
    for b in range(2):
        A32 = synth.spd_matrix(w, b).astype(np.float32)
        Ls, i_s = oracle.potrf_one(A32, uplo)
        Ld, i_d = oracle.dpotrf_one(A32.astype(np.float64), uplo)
        assert i_s == i_d == 0
        assert np.array_equal(Ls, Ld)


@pytest.mark.parametrize("k", [0, 5, 63])
def test_info_by_construction(k):
    w = synth.WORKLOADS["n64"]
    A = synth.make_indefinite(synth.spd_matrix(w, k), k, delta=1e-3)
    for uplo in ("L", "U"):
        _, info = oracle.dpotrf_one(A, uplo)
        assert info == k + 1


def test_batched_matches_single_and_ignores_the_other_triangle():
    n, lda, batch = 13, 15, 4
    mats = [synth.gram(n, synth.rng(44, b), "normal", float(n), 1.0) for b in range(batch)]
    for uplo in ("L", "U"):
        buf = np.full(batch * lda * n, np.nan)
        for b, M in enumerate(mats):
            for j in range(n):
                s0 = b * lda * n + j * lda
                if uplo == "L":
                    buf[s0 + j: s0 + n] = M[j:, j]
                else:
                    buf[s0: s0 + j + 1] = M[: j + 1, j]
        F, info, _ = oracle.dpotrf_batched(buf, n, lda, lda * n, batch, nthreads=2, uplo=uplo)
        assert not info.any()
        for b, M in enumerate(mats):
            want, _ = oracle.dpotrf_one(M, uplo)
            assert np.array_equal(F[b], want)
        F2, _, _ = oracle.dpotrf_batched(buf, n, lda, lda * n, batch, indices=[2], uplo=uplo)
        assert np.array_equal(F2[0], F[2])


def test_reconstruction_is_at_double_rounding():
    w = synth.WORKLOADS["n128"]
    A = synth.spd_matrix(w, 3)
    L, info = oracle.dpotrf_one(A)
    assert info == 0
    assert checks.recon_error(L, np.tril(A)) <= 10 * 128 * 2.0 ** -53


# --------------------------------------------------------------------------
# Planted mistakes
# --------------------------------------------------------------------------

MUTANTS = {
    "identity": ("", ""),
    "input rounded to float": ("double d = A[j + (int64_t)j * lda];",
                               "double d = (double)(float)A[j + (int64_t)j * lda];"),
    "off-diagonal rounded to float": ("double s = A[i + (int64_t)j * lda];",
                                      "double s = (double)(float)A[i + (int64_t)j * lda];"),
    "pivot sign": ("d -= ljk * ljk;", "d += ljk * ljk;"),
    "dropped update term": ("for (int k = 0; k < j; ++k)\n                s -= L",
                            "for (int k = 1; k < j; ++k)\n                s -= L"),
    "upper reads the lower triangle": ("double s = A[j + (int64_t)i * lda];",
                                       "double s = A[i + (int64_t)j * lda];"),
    "info zero-based": ("return j + 1;", "return j;"),
}


def _battery(lib) -> list[str]:
    for fn in (lib.oracle_dpotrf_one, lib.oracle_dpotrf_upper_one):
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]

    def run(fn, A):
        a = np.asfortranarray(np.asarray(A, dtype=np.float64))
        n = a.shape[0]
        F = np.zeros((n, n), order="F")
        info = fn(a.ctypes.data, n, n, F.ctypes.data, n)
        return np.ascontiguousarray(F), info

    failed = []
    L = _int_lower(12, 7, 2 ** 13)
    A = L @ L.T
    Ap = np.tril(A) + np.triu(np.full_like(A, 1e300), 1)
    F, info = run(lib.oracle_dpotrf_one, Ap)
    if info != 0 or not np.array_equal(F, L):
        failed.append("integer lower")
    Au = np.triu(A) + np.tril(np.full_like(A, 1e300), -1)
    F, info = run(lib.oracle_dpotrf_upper_one, Au)
    if info != 0 or not np.array_equal(F, L.T):
        failed.append("integer upper")
    w = synth.WORKLOADS["n64"]
    Ai = synth.make_indefinite(synth.spd_matrix(w, 9), 9, delta=1e-3)
    if run(lib.oracle_dpotrf_one, Ai)[1] != 10:
        failed.append("info")
    return failed


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    if old:
        assert old in src, name
        src = src.replace(old, new, 1)
    c, so = tmp_path / "d.c", tmp_path / "d.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(c), "-o", str(so), "-lm"], check=True)
    failed = _battery(ctypes.CDLL(str(so)))
    if name == "identity":
        assert failed == [], failed
    else:
        assert failed, f"planted mistake {name!r} passed every pin"
