"""Parity of batched SPOTRS / SPOSV (solve with the Cholesky factor) with the
CPU oracle, through the C-ABI (GPU).

Tolerances (derived from the arithmetic, FP32 unit roundoff u = 2^-24):
  * residual: ||B - L L^T X||_F / (||L||_F^2 ||X||_F) <= 2.38e-6 n. Each
    triangular solve in FP32 is backward stable with |dL| <= n u |L|, so the
    two solves leave a residual below about 2 n u ||L||^2 ||X||; 2.38e-6 n =
    20 u n (the factorization's printed budget) keeps a tenfold margin.
  * forward error against the oracle on the same FP32 factor:
    max|X - X_ref| / max|X_ref| <= 4 n u kappa_2(A), kappa_2(A) = kappa_2(L)^2
    computed in float64 (the perturbation bound of a backward-stable solve).
  * SPOSV: the residual against A, with the factorization's budget added:
    ||B - A X||_F / (||A||_F ||X||_F) <= 2 * 2.38e-6 n.
Everything outside the solution (the factor, B's padding rows and the gaps
between systems) must come back bitwise unchanged.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests import checks

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _built():
    from matrix_dense_linear_gb300 import build
    build.build()


def _factors(n, batch, seed, lda, strideA):
    """Oracle factors of gram matrices, rounded to FP32, lower triangles packed
    into a NaN-poisoned buffer (upper triangle, padding rows, gaps)."""
    mats = [synth.gram(n, synth.rng(seed, b), "normal", float(n), 1.0) for b in range(batch)]
    span = (batch - 1) * strideA + lda * n if batch else 0
    buf = np.full(max(span, 1), np.nan, dtype=np.float32)
    Ls = []
    for b, A in enumerate(mats):
        L, info = oracle.potrf_one(A)
        assert info == 0
        L32 = np.tril(L).astype(np.float32)
        Ls.append(L32)
        for j in range(n):
            buf[b * strideA + j * lda + j: b * strideA + j * lda + n] = L32[j:, j]
    return buf, Ls


def _rhs(n, nrhs, batch, seed, ldb, strideB):
    g = np.random.default_rng(seed)
    span = (batch - 1) * strideB + ldb * nrhs if batch else 0
    buf = np.full(max(span, 1), np.nan, dtype=np.float32)
    Bs = []
    for b in range(batch):
        B = g.standard_normal((n, nrhs)).astype(np.float32)
        Bs.append(B)
        for c in range(nrhs):
            buf[b * strideB + c * ldb: b * strideB + c * ldb + n] = B[:, c]
    return buf, Bs


def _solution_pattern(n, nrhs, ldb, strideB, batch, size):
    m = np.zeros(size, dtype=bool)
    for b in range(batch):
        for c in range(nrhs):
            m[b * strideB + c * ldb: b * strideB + c * ldb + n] = True
    return m


def _gpu_potrs(lbuf, n, lda, strideA, bbuf, nrhs, ldb, strideB, batch):
    import torch

    import matrix_dense_linear_gb300 as bl
    dl = torch.from_numpy(lbuf.copy()).cuda()
    db = torch.from_numpy(bbuf.copy()).cuda()
    code = bl.spotrs_batched(dl, n, lda, strideA, db, nrhs, ldb, strideB, batch)
    assert code == 0, code
    torch.cuda.synchronize()
    return dl.cpu().numpy(), db.cpu().numpy()


def _view(buf, n, nrhs, ldb, strideB, b):
    return np.stack([buf[b * strideB + c * ldb: b * strideB + c * ldb + n]
                     for c in range(nrhs)], axis=1)


def _check_solution(L32, B, X, X_ref, what):
    n = L32.shape[0]
    L = L32.astype(np.float64)
    Xd = X.astype(np.float64)
    res = np.linalg.norm(B.astype(np.float64) - L @ (L.T @ Xd))
    bound = checks.RECON_PER_N * n * np.linalg.norm(L) ** 2 * np.linalg.norm(Xd)
    assert res <= bound, f"{what}: residual {res:.3e} > {bound:.3e}"
    s = np.linalg.svd(L, compute_uv=False)
    kappa = (s[0] / s[-1]) ** 2
    err = np.abs(Xd - X_ref).max() / np.abs(X_ref).max()
    assert err <= 4 * n * U * kappa, f"{what}: forward error {err:.3e}, kappa {kappa:.1f}"


CASES = [(1, 1), (5, 3), (31, 8), (32, 32), (33, 33), (64, 1), (64, 2), (64, 70), (100, 17),
         (128, 32), (129, 40), (256, 16), (300, 5)]


@pytest.mark.parametrize("n,nrhs", CASES)
def test_potrs_parity(n, nrhs):
    batch = 5 if n <= 128 else 3
    lda, ldb = n + 3, n + 2
    strideA, strideB = lda * n + 5, ldb * nrhs + 7
    lbuf, Ls = _factors(n, batch, 900 + n, lda, strideA)
    bbuf, Bs = _rhs(n, nrhs, batch, 950 + n + nrhs, ldb, strideB)
    l_after, b_after = _gpu_potrs(lbuf, n, lda, strideA, bbuf, nrhs, ldb, strideB, batch)
    assert np.array_equal(l_after.view(np.uint32), lbuf.view(np.uint32)), "the factor changed"
    pat = _solution_pattern(n, nrhs, ldb, strideB, batch, bbuf.size)
    assert np.array_equal(b_after.view(np.uint32)[~pat], bbuf.view(np.uint32)[~pat]), \
        "memory outside the solutions changed"
    X_ref, _ = oracle.potrs_batched(lbuf, n, lda, strideA, bbuf, nrhs, ldb, strideB, batch)
    for b in range(batch):
        X = _view(b_after, n, nrhs, ldb, strideB, b)
        _check_solution(Ls[b], Bs[b], X, X_ref[b], f"n={n} nrhs={nrhs} system {b}")


@pytest.mark.parametrize("aligned", [True, False])
@pytest.mark.parametrize("n", [32, 97, 256, 300, 520, 1000])
def test_potrs_one_rhs_wavefront(n, aligned):
    """One right-hand side runs the wavefront form (a warp per 32-row block;
    8, 16 or 32 warps at most by n): every block size, the ragged last row
    block, and both forms of the L loads (16-byte ones when lda and the
    matrix stride are multiples of four floats, scalar ones otherwise)."""
    batch = 3
    if aligned:
        lda = (n + 3) // 4 * 4 + 4
        strideA, ldb, strideB = lda * n, n + 4, n + 8
    else:
        lda = n + 3
        strideA, ldb, strideB = lda * n + 5, n + 1, n + 3
    lbuf, Ls = _factors(n, batch, 1700 + n, lda, strideA)
    bbuf, Bs = _rhs(n, 1, batch, 1750 + n, ldb, strideB)
    l_after, b_after = _gpu_potrs(lbuf, n, lda, strideA, bbuf, 1, ldb, strideB, batch)
    assert np.array_equal(l_after.view(np.uint32), lbuf.view(np.uint32))
    pat = _solution_pattern(n, 1, ldb, strideB, batch, bbuf.size)
    assert np.array_equal(b_after.view(np.uint32)[~pat], bbuf.view(np.uint32)[~pat])
    X_ref, _ = oracle.potrs_batched(lbuf, n, lda, strideA, bbuf, 1, ldb, strideB, batch)
    for b in range(batch):
        _check_solution(Ls[b], Bs[b], _view(b_after, n, 1, ldb, strideB, b), X_ref[b],
                        f"n={n} aligned={aligned} system {b}")


@pytest.mark.parametrize("uplo", ["L", "U"])
@pytest.mark.parametrize("n,nrhs", [(32, 2), (40, 4), (61, 9), (64, 16)])
def test_potrs_register_form(n, nrhs, uplo):
    """Several right-hand sides up to n = 64 run the register form (a warp per
    system and group of up to eight right-hand sides, L blocks in registers):
    lda and the matrix stride multiples of four floats, so the L loads that are
    contiguous per lane take 16-byte accesses; both storages."""
    import torch

    import matrix_dense_linear_gb300 as bl
    batch = 4
    lda = (n + 3) // 4 * 4
    strideA, ldb, strideB = lda * n + 8, n + 1, (n + 1) * nrhs + 3
    lbuf, Ls = _factors(n, batch, 1800 + n, lda, strideA)
    if uplo == "U":  # the same factors as U = L^T in the upper triangle
        ubuf = np.full_like(lbuf, np.nan)
        for b in range(batch):
            for j in range(n):
                ubuf[b * strideA + j * lda: b * strideA + j * lda + j + 1] = Ls[b][j, : j + 1]
        lbuf = ubuf
    bbuf, Bs = _rhs(n, nrhs, batch, 1850 + n, ldb, strideB)
    dl = torch.from_numpy(lbuf.copy()).cuda()
    db = torch.from_numpy(bbuf.copy()).cuda()
    assert bl.spotrs_batched_uplo(uplo, dl, n, lda, strideA, db, nrhs, ldb, strideB, batch) == 0
    torch.cuda.synchronize()
    b_after = db.cpu().numpy()
    assert np.array_equal(dl.cpu().numpy().view(np.uint32), lbuf.view(np.uint32))
    pat = _solution_pattern(n, nrhs, ldb, strideB, batch, bbuf.size)
    assert np.array_equal(b_after.view(np.uint32)[~pat], bbuf.view(np.uint32)[~pat])
    X_ref, _ = oracle.potrs_batched(lbuf, n, lda, strideA, bbuf, nrhs, ldb, strideB, batch,
                                    uplo=uplo)
    for b in range(batch):
        _check_solution(Ls[b], Bs[b], _view(b_after, n, nrhs, ldb, strideB, b), X_ref[b],
                        f"n={n} nrhs={nrhs} {uplo} system {b}")


def test_potrs_large_order():
    n, nrhs, batch = 1024, 32, 2
    lbuf, Ls = _factors(n, batch, 1100, n, n * n)
    bbuf, Bs = _rhs(n, nrhs, batch, 1101, n, n * nrhs)
    _, b_after = _gpu_potrs(lbuf, n, n, n * n, bbuf, nrhs, n, n * nrhs, batch)
    X_ref, _ = oracle.potrs_batched(lbuf, n, n, n * n, bbuf, nrhs, n, n * nrhs, batch)
    for b in range(batch):
        _check_solution(Ls[b], Bs[b], _view(b_after, n, nrhs, n, n * nrhs, b), X_ref[b],
                        f"n=1024 system {b}")


def test_potrs_deterministic_and_position_invariant():
    n, nrhs, batch = 96, 24, 9
    lbuf, _ = _factors(n, batch, 1200, n, n * n)
    bbuf, _ = _rhs(n, nrhs, batch, 1201, n, n * nrhs)
    _, x1 = _gpu_potrs(lbuf, n, n, n * n, bbuf, nrhs, n, n * nrhs, batch)
    _, x2 = _gpu_potrs(lbuf, n, n, n * n, bbuf, nrhs, n, n * nrhs, batch)
    assert np.array_equal(x1.view(np.uint32), x2.view(np.uint32))
    b = 5
    _, one = _gpu_potrs(lbuf[b * n * n:(b + 1) * n * n], n, n, n * n,
                        bbuf[b * n * nrhs:(b + 1) * n * nrhs], nrhs, n, n * nrhs, 1)
    assert np.array_equal(one.view(np.uint32),
                          x1[b * n * nrhs:(b + 1) * n * nrhs].view(np.uint32))


@pytest.mark.parametrize("n,nrhs", [(32, 4), (64, 33), (128, 8), (200, 3)])
def test_sposv_parity_and_info(n, nrhs):
    import torch

    import matrix_dense_linear_gb300 as bl
    batch = 8
    mats = []
    for t in range(batch):
        A = synth.gram(n, synth.rng(1300 + n, t), "normal", float(n), 1.0)
        if t in (2, 5):
            A = synth.make_indefinite(A, [n // 3, n - 1][t == 5], delta=0.5)
        mats.append(A)
    bt = synth.pack(lambda b: mats[b], n, batch, fill="nan")
    ldb = n + 1
    bbuf, Bs = _rhs(n, nrhs, batch, 1400 + n, ldb, ldb * nrhs)
    dA = torch.from_numpy(bt.buf.copy()).cuda()
    dB = torch.from_numpy(bbuf.copy()).cuda()
    info = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    assert bl.sposv_batched(dA, n, bt.lda, bt.strideA, dB, nrhs, ldb, ldb * nrhs, batch,
                            info) == 0
    torch.cuda.synchronize()
    a_after, b_after, inf = dA.cpu().numpy(), dB.cpu().numpy(), info.cpu().numpy()
    _, info_ref, _ = oracle.potrf_batched(bt.buf, n, bt.lda, bt.strideA, batch)
    assert np.array_equal(inf, info_ref)
    pat = _solution_pattern(n, nrhs, ldb, ldb * nrhs, batch, bbuf.size)
    assert np.array_equal(b_after.view(np.uint32)[~pat], bbuf.view(np.uint32)[~pat])
    av = synth.strided_view(a_after, n, bt.lda, bt.strideA, batch)
    for b in range(batch):
        X = _view(b_after, n, nrhs, ldb, ldb * nrhs, b)
        if info_ref[b] != 0:
            assert np.array_equal(X.view(np.uint32), Bs[b].view(np.uint32)), \
                f"system {b} failed to factor but B changed"
            continue
        A = checks.sym_from_lower(np.tril(np.array(bt.view()[b])))
        Xd = X.astype(np.float64)
        res = np.linalg.norm(Bs[b].astype(np.float64) - A @ Xd)
        bound = 2 * checks.RECON_PER_N * n * np.linalg.norm(A) * np.linalg.norm(Xd)
        assert res <= bound, f"system {b}: residual {res:.3e} > {bound:.3e}"
        # the factor left in A is the one spotrf gives
        L = np.tril(np.array(av[b], dtype=np.float64))
        assert checks.recon_error(L, np.tril(np.array(bt.view()[b]))) <= checks.RECON_PER_N * n


def test_sposv_full_workload_sampled():
    """The n = 256 workload (4096 systems) with 16 right-hand sides each, in the
    benchmark's configuration; the oracle checks a sample of the systems."""
    import torch

    import matrix_dense_linear_gb300 as bl
    bt = synth.workload_batch("n256", fill="mirror", include_info=False)
    n, batch, nrhs = bt.n, bt.batch, 16
    bbuf, Bs = _rhs(n, nrhs, batch, 1500, n, n * nrhs)
    dA = torch.from_numpy(bt.buf.copy()).cuda()
    dB = torch.from_numpy(bbuf.copy()).cuda()
    info = torch.zeros(batch, dtype=torch.int32, device="cuda")
    assert bl.sposv_batched(dA, n, bt.lda, bt.strideA, dB, nrhs, n, n * nrhs, batch, info) == 0
    torch.cuda.synchronize()
    assert not info.cpu().numpy().any()
    a_after, b_after = dA.cpu().numpy(), dB.cpu().numpy()
    sample = list(range(0, batch, batch // 16))
    X_ref, _ = oracle.potrs_batched(a_after, n, n, n * n, bbuf, nrhs, n, n * nrhs, batch,
                                    indices=sample)
    av = synth.strided_view(a_after, n, n, n * n, batch)
    for t, b in enumerate(sample):
        L32 = np.tril(np.array(av[b]))
        _check_solution(L32, Bs[b], _view(b_after, n, nrhs, n, n * nrhs, b), X_ref[t],
                        f"n256 system {b}")


def test_quick_returns():
    import torch

    import matrix_dense_linear_gb300 as bl
    info = torch.full((4,), 9, dtype=torch.int32, device="cuda")
    A = torch.zeros(4, device="cuda")
    B = torch.full((4,), 3.0, device="cuda")
    assert bl.sposv_batched(A, 0, 1, 0, B, 2, 1, 2, 4, info) == 0
    torch.cuda.synchronize()
    assert info.cpu().tolist() == [0] * 4 and B.cpu().tolist() == [3.0] * 4
    assert bl.spotrs_batched(A, 2, 2, 4, B, 0, 2, 0, 1) == 0
    assert bl.spotrs_batched(A, 2, 2, 4, B, 1, 2, 2, 0) == 0
