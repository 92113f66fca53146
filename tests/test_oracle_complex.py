"""Pins of the complex Hermitian oracle (CPOTRF and ZPOTRF, A = L L^H, lower and upper)
against what the mathematics fixes (CPU only): the 2 x 2 closed form,
Gaussian-integer factors recovered bit for bit, leading minors for n <= 3,
exact info, the real oracle (pinned on its own) on real inputs, the
conjugate-transpose relation between the storages, and planted mistakes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import synth

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "cchol_ref.c")


def gaussian_factor(n: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    L = np.tril(g.integers(-3, 4, (n, n)) + 1j * g.integers(-3, 4, (n, n)), -1)
    L[np.diag_indices(n)] = g.integers(1, 5, n)
    return L.astype(np.complex128)


def hermitian_spd(n: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    G = g.standard_normal((n, n)) + 1j * g.standard_normal((n, n))
    A = G @ G.conj().T / n + np.eye(n)
    return 0.5 * (A + A.conj().T)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_two_by_two(seed):
    g = np.random.default_rng(seed)
    a, c = g.uniform(1, 4, 2)
    b = complex(g.uniform(-1, 1), g.uniform(-1, 1))
    A = np.array([[a, np.conj(b)], [b, c]], dtype=np.complex64).astype(np.complex128)
    L, info = oracle.cpotrf_one(A)
    assert info == 0
    l11 = np.sqrt(A[0, 0].real)
    l21 = A[1, 0] / l11
    want = np.array([[l11, 0], [l21, np.sqrt(A[1, 1].real - abs(l21) ** 2)]])
    np.testing.assert_allclose(L, want, rtol=1e-13)


@pytest.mark.parametrize("n", [1, 2, 7, 16, 33, 64])
def test_gaussian_integer_factor_exact(n):
    L = gaussian_factor(n, 40 + n)
    A = L @ L.conj().T
    assert np.abs(A.real).max() < 2 ** 24 and np.abs(A.imag).max() < 2 ** 24
    Lo, info = oracle.cpotrf_one(A)
    assert info == 0 and np.array_equal(Lo, L)
    # upper storage: poison the strict lower triangle, expect U = L^H
    Ap = np.triu(A) + np.tril(np.full(A.shape, 1e30 + 1e30j), -1)
    Uo, info = oracle.cpotrf_one(Ap, "U")
    assert info == 0 and np.array_equal(Uo, L.conj().T)


@pytest.mark.parametrize("name", ["n32", "n64"])
def test_real_inputs_match_the_real_oracle(name):
    A32 = synth.spd_matrix(synth.WORKLOADS[name], 1).astype(np.float32)
    Lr, ir = oracle.potrf_one(A32)
    Lc, ic = oracle.cpotrf_one(A32.astype(np.complex64))
    assert ir == ic == 0
    assert np.array_equal(Lc.real, Lr) and not Lc.imag.any()


@pytest.mark.parametrize("n", [5, 40])
def test_upper_is_the_conjugate_transpose_and_diag_imag_ignored(n):
    A = hermitian_spd(n, n).astype(np.complex64)
    L, i1 = oracle.cpotrf_one(A)
    U, i2 = oracle.cpotrf_one(A, "U")
    assert i1 == i2 == 0
    assert np.array_equal(U, L.conj().T)
    B = A.copy()
    B[np.diag_indices(n)] += 7j  # not read
    assert np.array_equal(oracle.cpotrf_one(B)[0], L)
    assert np.abs(L @ L.conj().T - A.astype(np.complex128)).max() <= 1e-12 * np.abs(A).max() * n


@pytest.mark.parametrize("n", [1, 2, 3])
def test_leading_minors(n):
    g = np.random.default_rng(70 + n)
    for t in range(20):
        if t % 3 == 0:
            M = g.standard_normal((n, n)) + 1j * g.standard_normal((n, n))
            A = M + M.conj().T
        else:
            A = hermitian_spd(n, 100 * n + t)
        A = A.astype(np.complex64).astype(np.complex128)
        A[np.diag_indices(n)] = A[np.diag_indices(n)].real
        dets = [1.0] + [np.linalg.det(A[:k, :k]).real for k in range(1, n + 1)]
        want_info = next((k for k in range(1, n + 1) if dets[k] <= 0), 0)
        L, info = oracle.cpotrf_one(A)
        assert info == want_info
        for j in range(1, (n if info == 0 else info - 1) + 1):
            assert L[j - 1, j - 1].real == pytest.approx(np.sqrt(dets[j] / dets[j - 1]),
                                                          rel=1e-9)


@pytest.mark.parametrize("k", [0, 9, 31])
def test_info_by_construction(k):
    n = 32
    A = hermitian_spd(n, 500 + k)
    if k > 0:
        a = A[:k, k]
        q = (a.conj() @ np.linalg.solve(A[:k, :k], a)).real
    else:
        q = 0.0
    A[k, k] = q - 0.5
    A = A.astype(np.complex64)
    for uplo in ("L", "U"):
        assert oracle.cpotrf_one(A, uplo)[1] == k + 1


def test_batched_matches_single():
    n, lda, batch = 9, 11, 5
    mats = [hermitian_spd(n, 900 + b).astype(np.complex64) for b in range(batch)]
    for uplo in ("L", "U"):
        buf = np.full(batch * lda * n, np.nan + 1j * np.nan, dtype=np.complex64)
        for b, M in enumerate(mats):
            for j in range(n):
                s0 = b * lda * n + j * lda
                if uplo == "L":
                    buf[s0 + j: s0 + n] = M[j:, j]
                else:
                    buf[s0: s0 + j + 1] = M[: j + 1, j]
        F, info, _ = oracle.cpotrf_batched(buf, n, lda, lda * n, batch, nthreads=2, uplo=uplo)
        assert not info.any()
        for b, M in enumerate(mats):
            assert np.array_equal(F[b], oracle.cpotrf_one(M, uplo)[0])


# --------------------------------------------------------------------------
# Double-precision complex input (ZPOTRF)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [2, 9, 40])
def test_z_gaussian_integer_factor_beyond_single(n):
    # entries up to 2^13: A's entries pass 2^24 (not complex64-exact) but every
    # intermediate stays an exact double integer
    g = np.random.default_rng(60 + n)
    L = np.tril(g.integers(-2 ** 13, 2 ** 13, (n, n)) + 1j * g.integers(-2 ** 13, 2 ** 13, (n, n)),
                -1)
    L[np.diag_indices(n)] = g.integers(1, 2 ** 13, n)
    A = L @ L.conj().T
    assert np.abs(A).max() > 2 ** 24
    for uplo, want in (("L", L), ("U", L.conj().T)):
        F, info = oracle.zpotrf_one(A, uplo)
        assert info == 0 and np.array_equal(F, want)


def test_z_matches_c_on_complex64_inputs():
    A = hermitian_spd(30, 7).astype(np.complex64)
    for uplo in ("L", "U"):
        assert np.array_equal(oracle.zpotrf_one(A.astype(np.complex128), uplo)[0],
                              oracle.cpotrf_one(A, uplo)[0])
    buf = np.concatenate([np.asfortranarray(A).ravel(order="F")] * 3)
    F, info, _ = oracle.cpotrf_batched(buf.astype(np.complex128), 30, 30, 900, 3)
    assert not info.any() and np.array_equal(F[2], oracle.cpotrf_one(A)[0])


# --------------------------------------------------------------------------
# Planted mistakes
# --------------------------------------------------------------------------

MUTANTS = {
    "identity": ("", ""),
    "missing conjugate": ("s -= L[i + (int64_t)k * ldl] * conj(L[j + (int64_t)k * ldl]);",
                          "s -= L[i + (int64_t)k * ldl] * L[j + (int64_t)k * ldl];"),
    "square instead of modulus": ("d -= creal(ljk) * creal(ljk) + cimag(ljk) * cimag(ljk);",
                                  "d -= creal(ljk * ljk);"),
    "upper without conjugate": ("s -= conj(U[k + (int64_t)j * ldu]) * U[k + (int64_t)i * ldu];",
                                "s -= U[k + (int64_t)j * ldu] * U[k + (int64_t)i * ldu];"),
    "upper reads the lower triangle": ("double complex s = ld_c(A, dbl, j + (int64_t)i * lda);",
                                       "double complex s = ld_c(A, dbl, i + (int64_t)j * lda);"),
    "info zero-based": ("return j + 1;", "return j;"),
    "double input rounded to float": (
        "return ((const double *)A)[2 * idx] + ((const double *)A)[2 * idx + 1] * I;",
        "return (float)((const double *)A)[2 * idx] + (float)((const double *)A)[2 * idx + 1] * I;"),
}


def _battery(lib) -> list[str]:
    for fn in (lib.oracle_cpotrf_one, lib.oracle_cpotrf_upper_one):
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]

    def run(fn, A):
        a = np.asfortranarray(np.asarray(A, dtype=np.complex64))
        n = a.shape[0]
        F = np.zeros((n, n), dtype=np.complex128, order="F")
        info = fn(a.ctypes.data, n, n, F.ctypes.data, n)
        return np.ascontiguousarray(F), info

    failed = []
    L = gaussian_factor(12, 3)
    A = L @ L.conj().T
    F, info = run(lib.oracle_cpotrf_one, np.tril(A))
    if info != 0 or not np.array_equal(F, L):
        failed.append("integer lower")
    Au = np.triu(A) + np.tril(np.full(A.shape, 1e30 + 1e30j), -1)
    F, info = run(lib.oracle_cpotrf_upper_one, Au)
    if info != 0 or not np.array_equal(F, L.conj().T):
        failed.append("integer upper")
    d = np.diag(np.array([1, 4, 0, 9], dtype=np.complex64))
    if run(lib.oracle_cpotrf_one, d)[1] != 3:
        failed.append("info")
    lib.oracle_zpotrf_one.restype = ctypes.c_int
    lib.oracle_zpotrf_one.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_int]
    g = np.random.default_rng(5)
    Lz = np.tril(g.integers(-2 ** 13, 2 ** 13, (8, 8)) + 1j * g.integers(-2 ** 13, 2 ** 13, (8, 8)), -1)
    Lz[np.diag_indices(8)] = g.integers(1, 2 ** 13, 8)
    az = np.asfortranarray(Lz @ Lz.conj().T)
    Fz = np.zeros((8, 8), dtype=np.complex128, order="F")
    if lib.oracle_zpotrf_one(az.ctypes.data, 8, 8, Fz.ctypes.data, 8) != 0 or \
            not np.array_equal(np.ascontiguousarray(Fz), Lz):
        failed.append("integer double complex")
    return failed


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    if old:
        assert old in src, name
        src = src.replace(old, new, 1)
    c, so = tmp_path / "c.c", tmp_path / "c.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(c), "-o", str(so), "-lm"], check=True)
    failed = _battery(ctypes.CDLL(str(so)))
    if name == "identity":
        assert failed == [], failed
    else:
        assert failed, f"planted mistake {name!r} passed every pin"
