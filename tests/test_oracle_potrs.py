"""Pins of the SPOTRS oracle (A X = B with A = L L^T) against what the
mathematics fixes (CPU only): closed forms, exact integer solutions, Cramer's
rule in exact rational arithmetic, a backward-error invariant, independence
from everything outside the lower triangle, and a LAPACK cross-check.
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _int_factor(n: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(seed)
    L = np.tril(g.integers(-3, 4, (n, n)), -1).astype(np.float64)
    L[np.diag_indices(n)] = g.integers(1, 5, n)
    return L


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("l,b", [(2.0, 8.0), (0.5, 1.0), (3.0, -9.0), (1e-3, 1e-6)])
def test_one_by_one(l, b):
    x = oracle.potrs_one(np.array([[l]]), np.array([b]))
    l32, b32 = float(np.float32(l)), float(np.float32(b))
    assert x[0] == pytest.approx(b32 / (l32 * l32), rel=1e-15)


@pytest.mark.parametrize("a,b,c", [(2.0, 1.0, 3.0), (1.0, -2.0, 0.5), (4.0, 0.0, 1.0)])
def test_two_by_two(a, b, c):
    # A = [[a^2, a b], [a b, b^2 + c^2]] for L = [[a, 0], [b, c]]; det A = a^2 c^2
    L = np.array([[a, 0.0], [b, c]])
    r = np.array([[1.0, -2.0], [0.5, 3.0]])
    X = oracle.potrs_one(L, r)
    A11, A21, A22 = a * a, a * b, b * b + c * c
    det = A11 * A22 - A21 * A21
    want = np.array([[A22 * r[0, k] - A21 * r[1, k] for k in range(2)],
                     [-A21 * r[0, k] + A11 * r[1, k] for k in range(2)]]) / det
    np.testing.assert_allclose(X, want, rtol=1e-14)


@pytest.mark.parametrize("n", [1, 5, 32])
def test_diagonal_factor(n):
    g = np.random.default_rng(n)
    d = g.uniform(0.5, 4.0, n).astype(np.float32).astype(np.float64)
    B = g.standard_normal((n, 3)).astype(np.float32).astype(np.float64)
    X = oracle.potrs_one(np.diag(d), B)
    np.testing.assert_allclose(X, B / (d * d)[:, None], rtol=1e-15)


# --------------------------------------------------------------------------
# Exact integer solutions: B = L L^T X with integer L and X is exact in
# float32, every intermediate (L^T X, then X) is an integer, so the oracle
# must give X bit for bit.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n,nrhs", [(1, 1), (2, 3), (7, 4), (16, 1), (33, 5), (64, 2)])
def test_integer_solution_exact(n, nrhs):
    L = _int_factor(n, 100 + n)
    g = np.random.default_rng(200 + n)
    X = g.integers(-5, 6, (n, nrhs)).astype(np.float64)
    B = L @ (L.T @ X)
    assert np.abs(B).max() < 2 ** 24  # exact in float32
    got = oracle.potrs_one(L, B)
    assert np.array_equal(got, X)


# --------------------------------------------------------------------------
# Brute force: Cramer's rule on A = L L^T in exact rationals (n <= 4)
# --------------------------------------------------------------------------

def _det(M):
    n = len(M)
    tot = Fraction(0)
    for perm in itertools.permutations(range(n)):
        sign = 1
        for i in range(n):
            for j in range(i + 1, n):
                if perm[i] > perm[j]:
                    sign = -sign
        p = Fraction(sign)
        for i in range(n):
            p *= M[i][perm[i]]
        tot += p
    return tot


@pytest.mark.parametrize("n", [1, 2, 3, 4])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_cramer(n, seed):
    g = np.random.default_rng(10 * n + seed)
    L = np.tril(g.standard_normal((n, n))).astype(np.float32)
    L[np.diag_indices(n)] = np.abs(L[np.diag_indices(n)]) + np.float32(0.5)
    b = g.standard_normal(n).astype(np.float32)
    Lq = [[Fraction(float(L[i, j])) if j <= i else Fraction(0) for j in range(n)]
          for i in range(n)]
    A = [[sum(Lq[i][k] * Lq[j][k] for k in range(n)) for j in range(n)] for i in range(n)]
    detA = _det(A)
    want = []
    for c in range(n):
        Ac = [[Fraction(float(b[i])) if j == c else A[i][j] for j in range(n)] for i in range(n)]
        want.append(float(_det(Ac) / detA))
    got = oracle.potrs_one(L, b)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-13)


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n,nrhs", [(8, 1), (64, 16), (200, 3)])
def test_backward_error(n, nrhs):
    g = np.random.default_rng(n)
    G = g.standard_normal((n, n))
    L = np.linalg.cholesky(G @ G.T / n + np.eye(n)).astype(np.float32).astype(np.float64)
    B = g.standard_normal((n, nrhs)).astype(np.float32).astype(np.float64)
    X = oracle.potrs_one(L, B)
    R = L @ (L.T @ X) - B
    eps = 2.0 ** -53
    assert np.linalg.norm(R) <= 10 * n * eps * np.linalg.norm(L) ** 2 * np.linalg.norm(X)


def test_reads_only_the_lower_triangle_and_the_rows_it_owns():
    n, nrhs, lda, ldb, batch = 9, 3, 12, 11, 4
    g = np.random.default_rng(5)
    Ls, Bs = [], []
    lbuf = np.full(batch * lda * n, np.nan, dtype=np.float32)
    bbuf = np.full(batch * ldb * nrhs, np.nan, dtype=np.float32)
    for b in range(batch):
        L = np.tril(g.standard_normal((n, n))) + 2 * np.eye(n)
        B = g.standard_normal((n, nrhs))
        Ls.append(L.astype(np.float32))
        Bs.append(B.astype(np.float32))
        for j in range(n):
            lbuf[b * lda * n + j * lda + j: b * lda * n + j * lda + n] = Ls[-1][j:, j]
        for c in range(nrhs):
            bbuf[b * ldb * nrhs + c * ldb: b * ldb * nrhs + c * ldb + n] = Bs[-1][:, c]
    X, _ = oracle.potrs_batched(lbuf, n, lda, lda * n, bbuf, nrhs, ldb, ldb * nrhs, batch,
                                nthreads=3)
    for b in range(batch):
        want = oracle.potrs_one(Ls[b], Bs[b])
        assert np.array_equal(X[b], want)
        assert np.isfinite(X[b]).all()


def test_batched_subset_matches_single():
    n, nrhs, batch = 17, 4, 6
    g = np.random.default_rng(8)
    Ls = [(np.tril(g.standard_normal((n, n))) + 3 * np.eye(n)).astype(np.float32)
          for _ in range(batch)]
    Bs = [g.standard_normal((n, nrhs)).astype(np.float32) for _ in range(batch)]
    lbuf = np.concatenate([L.T.ravel() for L in Ls])
    bbuf = np.concatenate([B.T.ravel() for B in Bs])
    X, _ = oracle.potrs_batched(lbuf, n, n, n * n, bbuf, nrhs, n, n * nrhs, batch,
                                indices=[4, 1])
    assert np.array_equal(X[0], oracle.potrs_one(Ls[4], Bs[4]))
    assert np.array_equal(X[1], oracle.potrs_one(Ls[1], Bs[1]))


def test_lapack_cross_check():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    n, nrhs = 50, 6
    g = np.random.default_rng(9)
    G = g.standard_normal((n, n))
    L = np.linalg.cholesky(G @ G.T / n + np.eye(n)).astype(np.float32).astype(np.float64)
    B = g.standard_normal((n, nrhs)).astype(np.float32).astype(np.float64)
    want = scipy_linalg.cho_solve((L, True), B)
    np.testing.assert_allclose(oracle.potrs_one(L, B), want, rtol=1e-12, atol=1e-13)
