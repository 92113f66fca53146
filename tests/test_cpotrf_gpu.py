"""Parity of the complex Hermitian factorizations (CPOTRF, ZPOTRF) with the
complex oracle, through the C-ABI (GPU).

CPOTRF takes the single-precision bars of the real path in complex
arithmetic: info bit-exact; max|L - L_oracle| / max|L_oracle| <= 1e-5 n; the
reconstruction ||L L^H - A||_F / ||A||_F <= 2.38e-6 n over the full Hermitian
matrix the stored triangle defines (diagonal: its real part). ZPOTRF takes
them rescaled from u32 = 2^-24 to u64 = 2^-53, the reconstruction evaluated
in extended precision. Everything outside the factored triangle
(NaN-poisoned) comes back bitwise unchanged; the diagonal's imaginary part
is not read.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests import checks

pytestmark = pytest.mark.gpu

U64, U32 = 2.0 ** -53, 2.0 ** -24
BARS = {"c64": (checks.MAXREL_PER_N, checks.RECON_PER_N),
        "c128": (checks.MAXREL_PER_N * U64 / U32, 20 * U64)}
DT = {"c64": np.complex64, "c128": np.complex128}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from matrix_dense_linear_gb300 import build
    build.build()


def _herm(n, seed):
    g = np.random.default_rng(seed)
    G = g.standard_normal((n, n)) + 1j * g.standard_normal((n, n))
    A = G @ G.conj().T / n + np.eye(n)
    return 0.5 * (A + A.conj().T)


def _pack(mats, n, lda, strideA, uplo, diag_imag=0.0, dt="c64"):
    batch = len(mats)
    buf = np.full(max((batch - 1) * strideA + lda * n, 1), np.nan + 1j * np.nan,
                  dtype=DT[dt])
    for b, M in enumerate(mats):
        M = np.array(M, dtype=DT[dt])
        M[np.diag_indices(n)] = M[np.diag_indices(n)].real + 1j * diag_imag
        for j in range(n):
            s0 = b * strideA + j * lda
            if uplo == "L":
                buf[s0 + j: s0 + n] = M[j:, j]
            else:
                buf[s0: s0 + j + 1] = M[: j + 1, j]
    return buf


def _pattern(n, lda, strideA, batch, size, uplo):
    m = np.zeros(size, dtype=bool)
    for b in range(batch):
        for j in range(n):
            s0 = b * strideA + j * lda
            if uplo == "L":
                m[s0 + j: s0 + n] = True
            else:
                m[s0: s0 + j + 1] = True
    return m


def _run(buf, n, lda, strideA, batch, uplo):
    import torch

    import matrix_dense_linear_gb300 as bl
    d = torch.from_numpy(buf.copy()).cuda()
    info = torch.full((max(batch, 1),), -7, dtype=torch.int32, device="cuda")
    bl.factor_complex(d, n, lda, strideA, batch, info, uplo=uplo)
    torch.cuda.synchronize()
    return d.cpu().numpy(), info.cpu().numpy()[:batch]


def _slot(buf, n, lda, strideA, b):
    s0 = b * strideA
    return np.stack([buf[s0 + j * lda: s0 + j * lda + n] for j in range(n)], axis=1)


def _check(buf, out, info, n, lda, strideA, batch, uplo, what):
    dt = "c128" if buf.dtype == np.complex128 else "c64"
    maxrel, recon = BARS[dt]
    pat = _pattern(n, lda, strideA, batch, buf.size, uplo)
    ov, bv = out.view(np.uint64), buf.view(np.uint64)
    if dt == "c128":  # two 64-bit words an element
        pat = np.repeat(pat, 2)
    assert np.array_equal(ov[~pat], bv[~pat]), what
    F, iref, _ = oracle.cpotrf_batched(buf, n, lda, strideA, batch, uplo=uplo)
    assert np.array_equal(info, iref), (what, info, iref)
    for b in range(batch):
        G = _slot(out, n, lda, strideA, b).astype(np.complex128)
        L = np.tril(G) if uplo == "L" else np.triu(G).conj().T
        R = F[b] if uplo == "L" else F[b].conj().T
        k = n if iref[b] == 0 else int(iref[b]) - 1
        if k == 0:
            continue
        e = np.abs(L[:k, :k] - R[:k, :k]).max() / np.abs(R[:k, :k]).max()
        assert e <= maxrel * k, (what, b, e)
        if iref[b]:
            continue
        Ain = _slot(buf, n, lda, strideA, b).astype(np.complex128)
        low = np.tril(Ain) if uplo == "L" else np.triu(Ain).conj().T
        Ah = np.tril(low, -1) + np.tril(low, -1).conj().T + np.diag(low.diagonal().real)
        assert np.abs(np.diag(L).imag).max() == 0.0, (what, b, "complex diagonal")
        if dt == "c64":
            r = np.linalg.norm(L @ L.conj().T - Ah) / np.linalg.norm(Ah)
        else:
            Lq, Aq = L.astype(np.clongdouble), Ah.astype(np.clongdouble)
            Rq = Lq @ Lq.conj().T - Aq
            r = float(np.sqrt((np.abs(Rq) ** 2).sum() / (np.abs(Aq) ** 2).sum()))
        assert r <= recon * n, (what, b, r)


@pytest.mark.parametrize("n", [1, 2, 5, 16, 31, 32, 33, 64, 100, 128, 129, 200, 256, 300])
@pytest.mark.parametrize("uplo", ["L", "U"])
@pytest.mark.parametrize("dt", ["c64", "c128"])
def test_cpotrf_parity(n, uplo, dt):
    batch = 6 if n <= 128 else 3
    mats = [_herm(n, 2000 + 10 * n + b) for b in range(batch)]
    for lda, strideA in ((n, n * n), (n + 3, (n + 3) * n + 5)):
        buf = _pack(mats, n, lda, strideA, uplo, diag_imag=0.25, dt=dt)
        out, info = _run(buf, n, lda, strideA, batch, uplo)
        _check(buf, out, info, n, lda, strideA, batch, uplo, f"n={n} lda={lda} {uplo}")


@pytest.mark.parametrize("n", [3, 8, 9, 16, 20, 32, 33, 48, 64, 65, 96, 97, 128])
@pytest.mark.parametrize("uplo", ["L", "U"])
def test_cpotrf_small_orders_ragged_batch(n, uplo):
    """Orders of the register kernels (several matrices a warp below 17, two
    warps a matrix above 32, a warp per 32 x 32 tile above 64) over a batch
    that leaves the last warp partly empty, with a padded lda and gaps."""
    batch = 301
    mats = [_herm(n, 3100 + 7 * n + b) for b in range(batch)]
    lda = n + 1
    strideA = lda * n + 3
    buf = _pack(mats, n, lda, strideA, uplo, diag_imag=-1.5)
    out, info = _run(buf, n, lda, strideA, batch, uplo)
    _check(buf, out, info, n, lda, strideA, batch, uplo, f"ragged n={n} {uplo}")


@pytest.mark.parametrize("n", [8, 20, 32, 64, 128, 200])
@pytest.mark.parametrize("dt", ["c64", "c128"])
def test_cpotrf_info(n, dt):
    g = np.random.default_rng(n)
    ks = [0, n - 1, n // 2, int(g.integers(0, n))]
    mats = [_herm(n, 2500 + 10 * n + b) for b in range(6)]
    for t, k in enumerate(ks):
        A = mats[t]
        q = (A[:k, k].conj() @ np.linalg.solve(A[:k, :k], A[:k, k])).real if k else 0.0
        A[k, k] = q - 0.5
    for uplo in ("L", "U"):
        buf = _pack(mats, n, n, n * n, uplo, dt=dt)
        out, info = _run(buf, n, n, n * n, 6, uplo)
        assert list(info[:4]) == [k + 1 for k in ks] and info[4] == 0 and info[5] == 0
        _check(buf, out, info, n, n, n * n, 6, uplo, f"info n={n} {uplo} {dt}")


def test_cpotrf_real_input_matches_spotrf():
    """A real symmetric matrix given as complex: the same factor as the
    single-precision real call, to within the tolerance (different kernels)."""
    import torch

    import matrix_dense_linear_gb300 as bl
    n, batch = 64, 8
    mats = [_herm(n, 2700 + b).real for b in range(batch)]
    bufc = _pack(mats, n, n, n * n, "L")
    outc, infoc = _run(bufc, n, n, n * n, batch, "L")
    bufr = np.concatenate([np.asfortranarray(M.astype(np.float32)).ravel(order="F") for M in mats])
    d = torch.from_numpy(bufr.copy()).cuda()
    info = torch.zeros(batch, dtype=torch.int32, device="cuda")
    bl.factor(d, n, n, n * n, batch, info)
    outr = d.cpu().numpy()
    assert not infoc.any() and not info.cpu().numpy().any()
    for b in range(batch):
        Lc = np.tril(_slot(outc, n, n, n * n, b))
        Lr = np.tril(_slot(outr, n, n, n * n, b))
        assert np.abs(Lc.imag).max() == 0.0
        assert np.abs(Lc.real - Lr).max() <= 2e-5 * n * np.abs(Lr).max()


def test_cpotrf_codes():
    import torch

    import matrix_dense_linear_gb300 as bl
    info = torch.full((3,), 9, dtype=torch.int32, device="cuda")
    A = torch.zeros(4, dtype=torch.complex64, device="cuda")
    assert bl.cpotrf_batched(A, 0, 1, 0, 3, info) == 0
    torch.cuda.synchronize()
    assert info.cpu().tolist() == [0] * 3
    assert bl.cpotrf_batched(A, 2, 1, 4, 1, info) == -3
    assert bl.cpotrf_batched(A, 2, 2, 4, 1, info, uplo="Z") == -1
    # a 4-byte-aligned (not 8) address is refused before any launch
    assert bl.cpotrf_batched(A.data_ptr() + 4, 2, 2, 4, 1, info) == -1
    assert bl.cpotrf_batched(A.data_ptr() + 4, 2, 2, 4, 1, info, uplo="U") == -2
    Z = torch.zeros(4, dtype=torch.complex128, device="cuda")
    assert bl.cpotrf_batched(Z.data_ptr() + 8, 2, 2, 4, 1, info, double=True) == -1
    assert bl.cpotrf_batched(Z, 2, 1, 4, 1, info) == -3


@pytest.mark.parametrize("uplo", ["L", "U"])
@pytest.mark.parametrize("n", [130, 256, 384, 520])
def test_cpotrf_tensor_core_update(n, uplo):
    """Single-precision complex, 16-byte-aligned batches above n = 128 (both
    storages): the panel solve's block updates and the trailing update run on
    the tensor cores (3xTF32 real and imaginary products); several row blocks
    and trailing tiles, ragged ones at 130 and 520; a padded lda."""
    batch = 5
    lda = n + 2
    mats = [_herm(n, 4000 + 10 * n + b) for b in range(batch)]
    buf = _pack(mats, n, lda, lda * n, uplo, diag_imag=0.75)
    out, info = _run(buf, n, lda, lda * n, batch, uplo)
    _check(buf, out, info, n, lda, lda * n, batch, uplo, f"tensor-core update n={n} {uplo}")


@pytest.mark.parametrize("uplo", ["L", "U"])
@pytest.mark.parametrize("cls", [6, 7])
def test_cpotrf_tensor_core_give_up(cls, uplo):
    """Classes 6 and 7 of the failure injection: the complex tensor-core
    trailing update (6) or panel solve (7) gives up at its first bounded wait
    for every third matrix: those report -1, the others match the oracle,
    nothing outside the triangles changes, and the next call factors the whole
    batch."""
    import matrix_dense_linear_gb300 as bl
    lib = bl.library()
    n, batch = 384, 6
    mats = [_herm(n, 4500 + b) for b in range(batch)]
    buf = _pack(mats, n, n, n * n, uplo)
    assert lib.bl_debug_fail_first_wait(cls, 3) == 0
    try:
        out, info = _run(buf, n, n, n * n, batch, uplo)
    finally:
        assert lib.bl_debug_fail_first_wait(cls, 0) == 0
    assert [int(x) for x in info] == [-1 if b % 3 == 0 else 0 for b in range(batch)], list(info)
    pat = _pattern(n, n, n * n, batch, buf.size, uplo)
    assert np.array_equal(out.view(np.uint64)[~pat], buf.view(np.uint64)[~pat])
    keep = [b for b in range(batch) if b % 3]
    sub = _pack([mats[b] for b in keep], n, n, n * n, uplo)
    sub_out = np.concatenate([out[b * n * n:(b + 1) * n * n] for b in keep])
    _check(sub, sub_out, np.zeros(len(keep), dtype=np.int32), n, n, n * n, len(keep), uplo,
           "give-up: untouched matrices")
    out2, info2 = _run(buf, n, n, n * n, batch, uplo)
    _check(buf, out2, info2, n, n, n * n, batch, uplo, "after the give-up")


@pytest.mark.parametrize("uplo", ["L", "U"])
def test_cpotrf_tensor_core_info(uplo):
    """Failed pivots in the later panels of the tensor-core complex path: the
    panel solve and the update skip a failed matrix, info is the oracle's and the
    leading block before the failure matches."""
    n = 384
    ks = [130, 300, 383, 5]
    mats = [_herm(n, 4700 + b) for b in range(6)]
    for t, k in enumerate(ks):
        A = mats[t]
        q = (A[:k, k].conj() @ np.linalg.solve(A[:k, :k], A[:k, k])).real
        A[k, k] = q - 0.5
    buf = _pack(mats, n, n, n * n, uplo)
    out, info = _run(buf, n, n, n * n, 6, uplo)
    assert list(info[:4]) == [k + 1 for k in ks] and info[4] == 0 and info[5] == 0, list(info)
    _check(buf, out, info, n, n, n * n, 6, uplo, "tensor-core info")
