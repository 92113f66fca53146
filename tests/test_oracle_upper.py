"""Pins of the uplo = 'U' oracle (A = U^T U from the upper triangle, and the
solve with U) against what the mathematics fixes (CPU only): closed forms,
exact integer factors and solutions, brute force by leading minors, reads of
the upper triangle only, and the relation U = L^T to the lower oracle, which
its own pins fix independently.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
import synth
from tests import checks
from tests.test_oracle import _brute


def _int_upper(n: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    U = np.triu(g.integers(-3, 4, (n, n)), 1).astype(np.float64)
    U[np.diag_indices(n)] = g.integers(1, 5, n)
    return U


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("a,info", [(4.0, 0), (2.0, 0), (0.0, 1), (-3.0, 1),
                                    (float("nan"), 1), (float("inf"), 0)])
def test_one_by_one(a, info):
    U, got = oracle.potrf_one(np.array([[a]]), uplo="U")
    assert got == info
    if info == 0:
        assert U[0, 0] == math.sqrt(float(np.float32(a)))


@pytest.mark.parametrize("a,b,c", [(4.0, 2.0, 5.0), (1.0, -0.5, 2.0), (9.0, 3.0, 1.5)])
def test_two_by_two_spd(a, b, c):
    # A = [[a, b], [b, c]]: U = [[sqrt a, b / sqrt a], [0, sqrt(c - b^2 / a)]]
    A = np.array([[a, b], [np.nan, c]])  # the strict lower triangle is never read
    U, info = oracle.potrf_one(A, uplo="U")
    assert info == 0
    ra = math.sqrt(a)
    want = np.array([[ra, b / ra], [0.0, math.sqrt(c - b * b / a)]])
    np.testing.assert_allclose(U, want, rtol=1e-15)


@pytest.mark.parametrize("a,b,c,info", [(1.0, 2.0, 3.0, 2), (1.0, 1.0, 1.0, 2), (-1.0, 0.0, 1.0, 1)])
def test_two_by_two_indefinite(a, b, c, info):
    _, got = oracle.potrf_one(np.array([[a, b], [b, c]]), uplo="U")
    assert got == info


def test_diagonal():
    d = np.array([4.0, 9.0, 0.0, 16.0], dtype=np.float32)
    U, info = oracle.potrf_one(np.diag(d), uplo="U")
    assert info == 3
    np.testing.assert_array_equal(np.diag(U)[:2], [2.0, 3.0])


# --------------------------------------------------------------------------
# Exact integer factors: A = U^T U with a small-integer U is exact in float32,
# and every intermediate of the oracle is an integer, so U comes back bit for
# bit.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 5, 16, 33, 100])
def test_integer_factor_is_recovered_exactly(n):
    U = _int_upper(n, 300 + n)
    A = U.T @ U
    assert np.abs(A).max() < 2 ** 24
    # the strict lower triangle carries garbage the oracle must not read
    Ap = np.triu(A) + np.tril(np.full((n, n), 1e30), -1)
    Uo, info = oracle.potrf_one(Ap, uplo="U")
    assert info == 0
    assert np.array_equal(Uo, U)


# --------------------------------------------------------------------------
# Brute force (leading minors, exact rationals) for n <= 4
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_brute_force_small(n):
    g = np.random.default_rng(500 + n)
    for trial in range(40):
        if trial % 3 == 0:
            A = g.standard_normal((n, n))
            A = A + A.T
        else:
            G = g.standard_normal((n, n))
            A = G @ G.T + 0.05 * np.eye(n)
        A32 = A.astype(np.float32)
        # the minors of the matrix the upper triangle defines: its transpose's
        # lower triangle
        Lb, ib = _brute(np.ascontiguousarray(A32.T))
        Uo, io = oracle.potrf_one(A32, uplo="U")
        assert io == ib
        m = n if ib == 0 else ib - 1
        if m:
            np.testing.assert_allclose(Uo[:m, :], Lb[:, :m].T, rtol=1e-9, atol=1e-12)


# --------------------------------------------------------------------------
# Relation to the lower oracle and invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["n32", "n64", "n128"])
def test_transpose_of_the_lower_factor_bit_for_bit(name):
    w = synth.WORKLOADS[name]
    for b in range(3):
        A32 = synth.spd_matrix(w, b).astype(np.float32)
        L, il = oracle.potrf_one(A32)
        U, iu = oracle.potrf_one(A32, uplo="U")
        assert il == iu == 0
        assert np.array_equal(U, L.T)
        assert checks.recon_error(U.T, np.tril(A32)) <= 1e-13


@pytest.mark.parametrize("k", [0, 7, 31])
def test_info_by_construction(k):
    w = synth.WORKLOADS["n32"]
    A32 = synth.make_indefinite(synth.spd_matrix(w, k), k).astype(np.float32)
    U, info = oracle.potrf_one(A32, uplo="U")
    assert info == k + 1
    L, il = oracle.potrf_one(A32)
    assert il == info
    assert np.array_equal(U[:k, :k], L[:k, :k].T)


def test_batched_reads_only_upper_triangles():
    n, lda, batch = 11, 13, 5
    w = synth.WORKLOADS["n32"]
    mats = [synth.gram(n, synth.rng(w.wid, b), "normal", float(n), 1.0).astype(np.float32)
            for b in range(batch)]
    buf = np.full(batch * lda * n, np.nan, dtype=np.float32)
    for b, M in enumerate(mats):
        for j in range(n):
            buf[b * lda * n + j * lda: b * lda * n + j * lda + j + 1] = M[: j + 1, j]
    F, info, _ = oracle.potrf_batched(buf, n, lda, lda * n, batch, nthreads=2, uplo="U")
    assert not info.any()
    for b, M in enumerate(mats):
        U, _ = oracle.potrf_one(M, uplo="U")
        assert np.array_equal(F[b], U)
        assert np.isfinite(F[b]).all()
    F2, _, _ = oracle.potrf_batched(buf, n, lda, lda * n, batch, indices=[3, 0], uplo="U")
    assert np.array_equal(F2[0], F[3]) and np.array_equal(F2[1], F[0])


def test_bad_uplo_is_rejected():
    with pytest.raises(ValueError):
        oracle.potrf_one(np.eye(2), uplo="X")


# --------------------------------------------------------------------------
# The solve with U: U^T U X = B
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n,nrhs", [(1, 1), (3, 2), (9, 4), (40, 3)])
def test_upper_solve_integer_exact(n, nrhs):
    U = _int_upper(n, 700 + n)
    X = np.random.default_rng(n).integers(-5, 6, (n, nrhs)).astype(np.float64)
    B = U.T @ (U @ X)
    assert np.abs(B).max() < 2 ** 24
    Up = U + np.tril(np.full((n, n), 1e30), -1)
    assert np.array_equal(oracle.potrs_one(Up, B, uplo="U"), X)


def test_upper_solve_matches_lower_solve_on_the_transpose():
    g = np.random.default_rng(12)
    n, nrhs = 37, 5
    G = g.standard_normal((n, n))
    L = np.linalg.cholesky(G @ G.T / n + np.eye(n)).astype(np.float32)
    B = g.standard_normal((n, nrhs)).astype(np.float32)
    assert np.array_equal(oracle.potrs_one(L.T, B, uplo="U"), oracle.potrs_one(L, B))


def test_upper_solve_batched():
    n, nrhs, batch, lda, ldb = 8, 3, 4, 10, 9
    g = np.random.default_rng(13)
    Us = [(np.triu(g.standard_normal((n, n))) + 3 * np.eye(n)).astype(np.float32)
          for _ in range(batch)]
    Bs = [g.standard_normal((n, nrhs)).astype(np.float32) for _ in range(batch)]
    lbuf = np.full(batch * lda * n, np.nan, dtype=np.float32)
    bbuf = np.full(batch * ldb * nrhs, np.nan, dtype=np.float32)
    for b in range(batch):
        for j in range(n):
            lbuf[b * lda * n + j * lda: b * lda * n + j * lda + j + 1] = Us[b][: j + 1, j]
        for c in range(nrhs):
            bbuf[b * ldb * nrhs + c * ldb: b * ldb * nrhs + c * ldb + n] = Bs[b][:, c]
    X, _ = oracle.potrs_batched(lbuf, n, lda, lda * n, bbuf, nrhs, ldb, ldb * nrhs, batch,
                                nthreads=2, uplo="U")
    for b in range(batch):
        assert np.array_equal(X[b], oracle.potrs_one(Us[b], Bs[b], uplo="U"))
