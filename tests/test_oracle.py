"""Pins of the CPU oracle against what the mathematics fixes (CPU only).

Each test checks the oracle against something other than itself: closed forms,
exact integer factors, brute force by Sylvester's criterion and bordered
minors in exact rational arithmetic, invariants, indefinite matrices with a
known failing pivot, and the pages' printed reconstruction budget.
"""
from __future__ import annotations

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from tests import checks


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("a,info", [(4.0, 0), (2.0, 0), (1e-30, 0), (0.0, 1), (-3.0, 1),
                                    (float("nan"), 1), (float("inf"), 0)])
def test_one_by_one(a, info):
    L, got = oracle.potrf_one(np.array([[a]]))
    assert got == info
    if info == 0:
        assert L[0, 0] == math.sqrt(np.float32(a))


@pytest.mark.parametrize("a,b,c", [(4.0, 2.0, 5.0), (2.0, -1.0, 3.0), (9.0, 3.0, 1.0000001),
                                   (1.0, 0.0, 1.0), (0.25, 0.125, 0.5)])
def test_two_by_two_spd(a, b, c):
    A = np.array([[a, b], [b, c]], dtype=np.float32).astype(np.float64)
    L, info = oracle.potrf_one(A)
    a, b, c = A[0, 0], A[1, 0], A[1, 1]
    assert info == 0
    assert L[0, 0] == pytest.approx(math.sqrt(a), rel=1e-15)
    assert L[1, 0] == pytest.approx(b / math.sqrt(a), rel=1e-15)
    assert L[1, 1] == pytest.approx(math.sqrt(c - b * b / a), rel=1e-12)
    assert L[0, 1] == 0.0


@pytest.mark.parametrize("a,b,c,info", [(1.0, 2.0, 3.0, 2), (1.0, 1.0, 1.0, 2), (4.0, 2.0, 0.5, 2),
                                        (-1.0, 0.0, 1.0, 1), (0.0, 1.0, 1.0, 1)])
def test_two_by_two_indefinite(a, b, c, info):
    # c - b^2/a <= 0 fails at pivot 2 even though every diagonal entry is positive
    _, got = oracle.potrf_one(np.array([[a, b], [b, c]]))
    assert got == info


@pytest.mark.parametrize("n", [1, 3, 8, 33])
def test_diagonal(n):
    g = np.random.default_rng(n)
    d = g.uniform(0.5, 9.0, n).astype(np.float32)
    L, info = oracle.potrf_one(np.diag(d))
    assert info == 0
    assert np.array_equal(np.diag(L), np.sqrt(d.astype(np.float64)))
    assert np.count_nonzero(L - np.diag(np.diag(L))) == 0
    for bad in range(n):
        for v in (0.0, -1.0, np.nan):
            dd = d.copy()
            dd[bad] = v
            if bad + 1 < n:
                dd[bad + 1] = -2.0  # a later failure must not win
            _, info = oracle.potrf_one(np.diag(dd))
            assert info == bad + 1


def test_hand_example_3x3():
    # L = [[3,0,0],[-1,2,0],[2,1,4]] gives A = L L^T = [[9,-3,6],[-3,5,0],[6,0,21]]
    A = np.array([[9, -3, 6], [-3, 5, 0], [6, 0, 21]], dtype=np.float64)
    L, info = oracle.potrf_one(A)
    assert info == 0
    assert np.array_equal(L, np.array([[3, 0, 0], [-1, 2, 0], [2, 1, 4]], dtype=np.float64))
    # same leading 2x2 block, a_33 lowered from 21 to 4: pivot 3 is 4 - 4 - 1 = -1
    A[2, 2] = 4.0
    assert oracle.potrf_one(A)[1] == 3


# --------------------------------------------------------------------------
# Exact recovery of an integer factor
# --------------------------------------------------------------------------

def _integer_factor(n: int, seed: int) -> np.ndarray:
    g = np.random.default_rng(1000 + seed)
    L = np.tril(g.integers(-3, 4, (n, n)), -1)
    L[np.diag_indices(n)] = g.integers(1, 5, n)
    return L.astype(np.int64)


@pytest.mark.parametrize("n", [1, 2, 5, 16, 33, 100, 257])
def test_integer_factor_is_recovered_exactly(n):
    L = _integer_factor(n, n)
    A = L @ L.T
    assert np.abs(A).max() < 2 ** 24  # exact in float32
    Lo, info = oracle.potrf_one(A.astype(np.float64))
    assert info == 0
    assert np.array_equal(Lo, L.astype(np.float64)), "integer L not reproduced bit-exactly"


# --------------------------------------------------------------------------
# Brute force for n <= 4: Sylvester's criterion and bordered minors, exact
# --------------------------------------------------------------------------

def _det(M):
    """Determinant by permutation expansion over Fractions."""
    n = len(M)
    tot = Fraction(0)
    for perm in itertools.permutations(range(n)):
        inv = sum(1 for i in range(n) for j in range(i + 1, n) if perm[i] > perm[j])
        p = Fraction(1)
        for i in range(n):
            p *= M[i][perm[i]]
        tot += -p if inv % 2 else p
    return tot


def _brute(A32: np.ndarray):
    """(L as float64, info) from leading minors: info = first k with det A_k <= 0,
    l_jj = sqrt(det A_j / det A_{j-1}),
    l_ij = det(A[{1..j-1, i}, {1..j}]) / sqrt(det A_j det A_{j-1})."""
    n = A32.shape[0]
    F = [[Fraction(float(A32[max(i, j), min(i, j)])) for j in range(n)] for i in range(n)]
    dets = [Fraction(1)]
    for k in range(1, n + 1):
        dets.append(_det([row[:k] for row in F[:k]]))
    info = 0
    for k in range(1, n + 1):
        if dets[k] <= 0:
            info = k
            break
    L = np.zeros((n, n))
    m = n if info == 0 else info - 1
    for j in range(1, m + 1):
        L[j - 1, j - 1] = math.sqrt(dets[j] / dets[j - 1])
        for i in range(j + 1, n + 1):
            rows = list(range(j - 1)) + [i - 1]
            num = _det([[F[r][c] for c in range(j)] for r in rows])
            L[i - 1, j - 1] = float(num) / math.sqrt(float(dets[j]) * float(dets[j - 1]))
    return L, info


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_brute_force_small(n):
    g = np.random.default_rng(77 + n)
    for trial in range(60):
        if trial % 3 == 0:
            A = g.standard_normal((n, n))  # mostly indefinite
            A = A + A.T
        else:
            G = g.standard_normal((n, n))
            A = G @ G.T + 0.05 * np.eye(n)
        A32 = A.astype(np.float32)
        Lb, ib = _brute(A32)
        Lo, io = oracle.potrf_one(A32)
        assert io == ib, (trial, A32)
        m = n if ib == 0 else ib - 1
        if m:
            np.testing.assert_allclose(Lo[:, :m], Lb[:, :m], rtol=1e-9, atol=1e-12)


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["n32", "n64", "n128"])
def test_invariants_on_workloads(name):
    w = synth.WORKLOADS[name]
    for b in (0, 7, w.batch - 1):
        A32 = synth.spd_matrix(w, b).astype(np.float32)
        L, info = oracle.potrf_one(A32)
        assert info == 0
        assert np.all(np.triu(L, 1) == 0)
        assert np.all(np.diag(L) > 0)
        r = checks.recon_error(L, np.tril(A32))
        assert r <= 10 * w.n * 2.0 ** -53 * 8, r


def test_upper_triangle_and_padding_are_ignored():
    w = synth.WORKLOADS["n32"]
    mats = [synth.workload_matrix(w, b) for b in range(8)] + \
           [synth.workload_matrix(w, w.batch + t) for t in range(4)]
    outs = []
    for fill in ("mirror", "nan", "big"):
        bt = synth.pack(lambda b: mats[b], 32, len(mats), lda=37, strideA=37 * 32 + 5, fill=fill)
        L, info, _ = oracle.potrf_batched(bt.buf, bt.n, bt.lda, bt.strideA, bt.batch)
        outs.append((L, info))
    for L, info in outs[1:]:
        assert np.array_equal(info, outs[0][1])
        assert np.array_equal(L, outs[0][0])


def test_batched_matches_single_and_thread_count():
    w = synth.WORKLOADS["n64"]
    bt = synth.pack(lambda b: synth.spd_matrix(w, b), 64, 9, fill="nan")
    L1, i1, _ = oracle.potrf_batched(bt.buf, 64, 64, 64 * 64, 9, nthreads=1)
    L4, i4, used = oracle.potrf_batched(bt.buf, 64, 64, 64 * 64, 9, nthreads=4)
    assert used == 4
    assert np.array_equal(L1, L4) and np.array_equal(i1, i4)
    for b in range(9):
        Ls, _ = oracle.potrf_one(bt.view()[b])
        assert np.array_equal(Ls, L1[b])
    Lsub, isub, _ = oracle.potrf_batched(bt.buf, 64, 64, 64 * 64, 9, indices=[8, 3])
    assert np.array_equal(Lsub[0], L1[8]) and np.array_equal(Lsub[1], L1[3])


# --------------------------------------------------------------------------
# Exact info by construction
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["n32", "n64", "n128"])
def test_info_by_construction(name):
    w = synth.WORKLOADS[name]
    g = np.random.default_rng(5)
    ks = sorted({0, 1, w.n // 2, w.n - 1, *g.integers(0, w.n, 4).tolist()})
    for k in ks:
        A = synth.make_indefinite(synth.spd_matrix(w, k), k)
        A32 = A.astype(np.float32)
        # the diagonal itself stays positive in most cases: a test on a_kk alone would fail
        L, info = oracle.potrf_one(A32)
        assert info == k + 1, (k, info)
        if k:
            Lref, _ = oracle.potrf_one(synth.spd_matrix(w, k).astype(np.float32))
            np.testing.assert_array_equal(L[:, :k], Lref[:, :k])


def test_info_matrices_of_the_n32_workload():
    w = synth.WORKLOADS["n32"]
    mats = [synth.workload_matrix(w, w.batch + t) for t in range(w.extra_info)]
    ks = [synth.info_pivot(w, t) for t in range(w.extra_info)]
    assert 0 in ks and w.n - 1 in ks
    for A, k in zip(mats, ks):
        assert oracle.potrf_one(A.astype(np.float32))[1] == k + 1


def test_failing_pivot_behind_a_positive_diagonal():
    # a small margin keeps a_kk > 0 while the Schur complement at k is negative:
    # an oracle that tested the raw diagonal instead of the pivot would miss it
    w = synth.WORKLOADS["n64"]
    seen = 0
    for k in (5, 20, 40, 63):
        A32 = synth.make_indefinite(synth.spd_matrix(w, k), k, delta=0.05).astype(np.float32)
        if A32[k, k] > 0:
            seen += 1
        assert oracle.potrf_one(A32)[1] == k + 1
    assert seen > 0


# --------------------------------------------------------------------------
# Library cross-check and the printed budget
# --------------------------------------------------------------------------

def test_lapack_cross_check():
    # LAPACK is a cross-check only, used where it passes its own residual check
    g = np.random.default_rng(3)
    for n in (5, 40, 130):
        G = g.standard_normal((n, n))
        A32 = (G @ G.T / n + np.eye(n)).astype(np.float32)
        A = A32.astype(np.float64)
        Ll = np.linalg.cholesky(A)
        if np.linalg.norm(Ll @ Ll.T - A) / np.linalg.norm(A) > 1e-13:
            continue
        Lo, info = oracle.potrf_one(A32)
        assert info == 0
        np.testing.assert_allclose(Lo, Ll, rtol=1e-11, atol=1e-13)


def test_printed_budget_is_twenty_flt_epsilon():
    assert checks.RECON_PER_N == pytest.approx(20 * 2.0 ** -23, rel=2e-3)
    assert checks.TOL["flt_epsilon_multiple"] == 20


def test_tolerance_separates_fp32_rounding_from_a_dropped_term():
    """The budget admits fp32 rounding but not a plausible bug: rounding the
    oracle's factor to float32 passes; dropping one product term fails."""
    w = synth.WORKLOADS["n64"]
    A32 = synth.spd_matrix(w, 1).astype(np.float32)
    L, _ = oracle.potrf_one(A32)
    assert checks.recon_error(L.astype(np.float32), np.tril(A32)) <= checks.RECON_PER_N * 64
    Lbad = L.copy()
    Lbad[40, 30] = 0.0  # one dropped entry
    assert checks.recon_error(Lbad, np.tril(A32)) > checks.RECON_PER_N * 64
    Lsign = L.copy()
    Lsign[50, 7] = -Lsign[50, 7]
    assert checks.recon_error(Lsign, np.tril(A32)) > checks.RECON_PER_N * 64
