"""Parity of the uplo = 'U' path (A = U^T U, the factor in the upper
triangle) with the CPU oracle, through the C-ABI (GPU).

The same bars as the lower path: info bit-exact; U against the oracle's U
within max|U - U_oracle| / max|U_oracle| <= 1e-5 n; the reconstruction
||U^T U - A||_F / ||A||_F within 2.38e-6 n; every element outside the upper
triangles (the strict lower triangle, rows n..lda-1, the gaps, all poisoned)
bitwise unchanged. Beyond the oracle: the kernels run the same arithmetic
with transposed addresses, so U must equal the transpose of the lower path's
L bit for bit wherever both take the same kernels.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests import checks

pytestmark = pytest.mark.gpu

WARP, CTA, BLOCKED, TMEM = 1, 2, 3, 4
U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _built():
    from matrix_dense_linear_gb300 import build
    build.build()


def _mats(n, batch, seed):
    return [synth.gram(n, synth.rng(seed, b), "normal", float(n), 1.0) for b in range(batch)]


def _pack_upper(mats, n, lda, strideA, poison=np.nan, offset=0):
    """Upper triangles (rounded once to FP32) in a poisoned buffer; returns
    (buffer with the offset in front, the offset)."""
    batch = len(mats)
    span = (batch - 1) * strideA + lda * n if batch else 0
    buf = np.full(offset + max(span, 1), poison, dtype=np.float32)
    for b, A in enumerate(mats):
        A32 = np.asarray(A).astype(np.float32)
        for j in range(n):
            s = offset + b * strideA + j * lda
            buf[s: s + j + 1] = A32[: j + 1, j]
    return buf


def _pack_lower(mats, n, lda, strideA, poison=np.nan):
    batch = len(mats)
    span = (batch - 1) * strideA + lda * n if batch else 0
    buf = np.full(max(span, 1), poison, dtype=np.float32)
    for b, A in enumerate(mats):
        A32 = np.asarray(A).astype(np.float32)
        for j in range(n):
            buf[b * strideA + j * lda + j: b * strideA + j * lda + n] = A32[j:, j]
    return buf


def _upper_pattern(n, lda, strideA, batch, size, offset=0):
    """True where an element belongs to an upper triangle."""
    m = np.zeros(size, dtype=bool)
    for b in range(batch):
        for j in range(n):
            s = offset + b * strideA + j * lda
            m[s: s + j + 1] = True
    return m


def _factor(buf, n, lda, strideA, batch, route=0, uplo="U", offset=0):
    import torch

    import matrix_dense_linear_gb300 as bl
    d = torch.from_numpy(buf.copy()).cuda()
    info = torch.full((max(batch, 1),), -7, dtype=torch.int32, device="cuda")
    ptr = d.data_ptr() + 4 * offset
    if uplo == "U":
        code = bl.spotrf_batched_uplo("U", ptr, n, lda, strideA, batch, info, None, route)
    else:
        code = bl.spotrf_batched_ex(ptr, n, lda, strideA, batch, info, None, route)
    assert code == 0, code
    torch.cuda.synchronize()
    return d.cpu().numpy(), info.cpu().numpy()[:batch]


def _slot(buf, n, lda, strideA, b, offset=0):
    s = offset + b * strideA
    return np.stack([buf[s + j * lda: s + j * lda + n] for j in range(n)], axis=1)  # [i, j]


def _check(buf_in, out, info, n, lda, strideA, batch, idx, what, offset=0):
    pat = _upper_pattern(n, lda, strideA, batch, buf_in.size, offset)
    bad = np.count_nonzero(out.view(np.uint32)[~pat] != buf_in.view(np.uint32)[~pat])
    assert bad == 0, f"{what}: {bad} elements outside the upper triangles changed"
    F, info_ref, _ = oracle.potrf_batched(buf_in[offset:], n, lda, strideA, batch,
                                          indices=idx, uplo="U")
    for t, b in enumerate(idx):
        Ug = np.triu(_slot(out, n, lda, strideA, b, offset))
        A_up = np.triu(_slot(buf_in, n, lda, strideA, b, offset))
        checks.check_factor(Ug.T, F[t].T, int(info[b]), int(info_ref[t]), A_up.T,
                            what=f"{what} matrix {b}")
    return info_ref


def _routes(n):
    r = [0, BLOCKED]
    if n <= 64:
        r.append(WARP)
    if n <= 128:
        r.append(CTA)
    else:
        r.append(5)  # the left-looking schedule
    return sorted(set(r))


@pytest.mark.parametrize("n", [1, 2, 5, 8, 16, 17, 31, 32, 33, 48, 63, 64, 65, 96, 100, 127,
                               128, 129, 200, 256, 300])
def test_upper_every_route(n):
    batch = 7 if n <= 128 else 3
    mats = _mats(n, batch, 900 + n)
    for lda, strideA in ((n, n * n), (n + 3, (n + 3) * n + 5)):
        buf = _pack_upper(mats, n, lda, strideA, poison=np.nan if n % 2 else np.float32(1e30))
        for route in _routes(n):
            out, info = _factor(buf, n, lda, strideA, batch, route)
            _check(buf, out, info, n, lda, strideA, batch, list(range(batch)),
                   f"U n={n} lda={lda} route={route}")


def test_upper_misaligned_base():
    n, batch = 40, 5
    mats = _mats(n, batch, 950)
    buf = _pack_upper(mats, n, n, n * n, offset=1)
    for route in (0, CTA, BLOCKED):
        out, info = _factor(buf, n, n, n * n, batch, route, offset=1)
        _check(buf, out, info, n, n, n * n, batch, list(range(batch)), f"U offset route={route}",
               offset=1)


@pytest.mark.parametrize("n,batch", [(48, 2000), (64, 1000), (32, 4096)])
def test_upper_large_batch_sampled(n, batch):
    """The batch sizes that take the one-warp kernel at n = 33 .. 64 (above
    four two-warp blocks per SM) and four-warp blocks at n <= 32."""
    mats = _mats(n, 64, 960 + n)
    buf = _pack_upper([mats[b % 64] for b in range(batch)], n, n, n * n)
    out, info = _factor(buf, n, n, n * n, batch)
    _check(buf, out, info, n, n, n * n, batch, [0, 1, 63, batch // 2, batch - 1],
           f"U n={n} batch={batch}")
    assert not info.any()


@pytest.mark.parametrize("n", [4, 32, 64, 100, 200])
def test_upper_info(n):
    g = np.random.default_rng(n + 7)
    ks = [0, n - 1, n // 2, int(g.integers(0, n))]
    mats = _mats(n, 8, 970 + n)
    for t, k in enumerate(ks):
        mats[t] = synth.make_indefinite(mats[t], k, delta=0.5)
    mats[5][:] = 0.0
    mats[6][0, 0] = -1.0
    buf = _pack_upper(mats, n, n, n * n)
    for route in _routes(n):
        out, info = _factor(buf, n, n, n * n, 8, route)
        info_ref = _check(buf, out, info, n, n, n * n, 8, list(range(8)), f"U n={n} route={route}")
        assert list(info_ref[:4]) == [k + 1 for k in ks]
        assert info_ref[5] == 1 and info_ref[6] == 1 and info_ref[7] == 0


@pytest.mark.parametrize("n,route,lda", [(20, WARP, 20), (48, WARP, 48), (64, WARP, 64),
                                         (100, CTA, 100), (128, CTA, 128), (200, BLOCKED, 203),
                                         (200, BLOCKED, 200), (384, BLOCKED, 388)])
def test_upper_is_the_lower_transposed_bit_for_bit(n, route, lda):
    """Same kernels, transposed addresses: U = L^T exactly, on the FP32 panel
    kernels (lda not a multiple of 4) and on the tensor-core ones."""
    batch = 9
    mats = _mats(n, batch, 990 + n)
    up = _pack_upper(mats, n, lda, lda * n)
    lo = _pack_lower(mats, n, lda, lda * n)
    out_u, info_u = _factor(up, n, lda, lda * n, batch, route, "U")
    out_l, info_l = _factor(lo, n, lda, lda * n, batch, route, "L")
    assert np.array_equal(info_u, info_l) and not info_u.any()
    for b in range(batch):
        Ug = np.triu(_slot(out_u, n, lda, lda * n, b))
        Lg = np.tril(_slot(out_l, n, lda, lda * n, b))
        assert np.array_equal(Ug.T.view(np.uint32), Lg.view(np.uint32)), f"matrix {b}"


def test_upper_tmem_route_refused_and_bad_uplo():
    import torch

    import matrix_dense_linear_gb300 as bl
    d = torch.zeros(64 * 64, device="cuda")
    info = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert bl.spotrf_batched_uplo("U", d, 64, 64, 64 * 64, 1, info, None, TMEM) == -9
    assert bl.spotrf_batched_uplo("X", d, 64, 64, 64 * 64, 1, info) == -1
    assert bl.spotrf_batched_uplo("u", d, 0, 1, 1, 1, info) == 0
    torch.cuda.synchronize()
    assert int(info[0]) == 0


# --------------------------------------------------------------------------
# The solve with U (bl_spotrs_batched_uplo, bl_sposv_batched_uplo)
# --------------------------------------------------------------------------

def _rhs(n, nrhs, batch, seed, ldb, strideB):
    g = np.random.default_rng(seed)
    buf = np.full(max((batch - 1) * strideB + ldb * nrhs, 1), np.nan, dtype=np.float32)
    Bs = []
    for b in range(batch):
        B = g.standard_normal((n, nrhs)).astype(np.float32)
        Bs.append(B)
        for c in range(nrhs):
            buf[b * strideB + c * ldb: b * strideB + c * ldb + n] = B[:, c]
    return buf, Bs


def _sol(buf, n, nrhs, ldb, strideB, b):
    return np.stack([buf[b * strideB + c * ldb: b * strideB + c * ldb + n]
                     for c in range(nrhs)], axis=1)


@pytest.mark.parametrize("n,nrhs", [(1, 1), (7, 3), (32, 8), (33, 17), (64, 40), (130, 5)])
def test_upper_solve_parity(n, nrhs):
    import torch

    import matrix_dense_linear_gb300 as bl
    batch, lda, ldb = 5, n + 2, n + 1
    strideA, strideB = lda * n + 3, ldb * nrhs + 2
    Us = []
    for A in _mats(n, batch, 1100 + n):
        Uo, info = oracle.potrf_one(A, uplo="U")
        assert info == 0
        Us.append(np.triu(Uo).astype(np.float32))
    ubuf = _pack_upper(Us, n, lda, strideA)  # U's upper triangle, poison elsewhere
    bbuf, Bs = _rhs(n, nrhs, batch, 1200 + n, ldb, strideB)
    du = torch.from_numpy(ubuf.copy()).cuda()
    db = torch.from_numpy(bbuf.copy()).cuda()
    assert bl.spotrs_batched_uplo("U", du, n, lda, strideA, db, nrhs, ldb, strideB, batch) == 0
    torch.cuda.synchronize()
    assert np.array_equal(du.cpu().numpy().view(np.uint32), ubuf.view(np.uint32))
    out = db.cpu().numpy()
    X_ref, _ = oracle.potrs_batched(ubuf, n, lda, strideA, bbuf, nrhs, ldb, strideB, batch,
                                    uplo="U")
    for b in range(batch):
        X = _sol(out, n, nrhs, ldb, strideB, b).astype(np.float64)
        Ud = Us[b].astype(np.float64)
        res = np.linalg.norm(Bs[b].astype(np.float64) - Ud.T @ (Ud @ X))
        bound = checks.RECON_PER_N * n * np.linalg.norm(Ud) ** 2 * np.linalg.norm(X)
        assert res <= bound, f"n={n} b={b}: residual {res:.3e} > {bound:.3e}"
        s = np.linalg.svd(Ud, compute_uv=False)
        err = np.abs(X - X_ref[b]).max() / np.abs(X_ref[b]).max()
        assert err <= 4 * n * U * (s[0] / s[-1]) ** 2
    # nothing but the solutions changed
    pat = np.zeros(bbuf.size, dtype=bool)
    for b in range(batch):
        for c in range(nrhs):
            pat[b * strideB + c * ldb: b * strideB + c * ldb + n] = True
    assert np.array_equal(out.view(np.uint32)[~pat], bbuf.view(np.uint32)[~pat])


@pytest.mark.parametrize("aligned", [True, False])
@pytest.mark.parametrize("n", [97, 300, 700])
def test_upper_solve_one_rhs(n, aligned):
    """One right-hand side with U (the wavefront form, 8, 16 and 32 warps at
    most): U's rows are contiguous there, so the forward pass reads them with
    16-byte loads when lda and the stride are multiples of four floats."""
    import torch

    import matrix_dense_linear_gb300 as bl
    batch = 3
    if aligned:
        lda = (n + 3) // 4 * 4
        strideA, ldb, strideB = lda * n + 4, n, n + 4
    else:
        lda = n + 1
        strideA, ldb, strideB = lda * n + 3, n + 2, n + 5
    Us = []
    for A in _mats(n, batch, 1300 + n):
        Uo, info = oracle.potrf_one(A, uplo="U")
        assert info == 0
        Us.append(np.triu(Uo).astype(np.float32))
    ubuf = _pack_upper(Us, n, lda, strideA)
    bbuf, Bs = _rhs(n, 1, batch, 1350 + n, ldb, strideB)
    du = torch.from_numpy(ubuf.copy()).cuda()
    db = torch.from_numpy(bbuf.copy()).cuda()
    assert bl.spotrs_batched_uplo("U", du, n, lda, strideA, db, 1, ldb, strideB, batch) == 0
    torch.cuda.synchronize()
    assert np.array_equal(du.cpu().numpy().view(np.uint32), ubuf.view(np.uint32))
    out = db.cpu().numpy()
    X_ref, _ = oracle.potrs_batched(ubuf, n, lda, strideA, bbuf, 1, ldb, strideB, batch,
                                    uplo="U")
    for b in range(batch):
        X = _sol(out, n, 1, ldb, strideB, b).astype(np.float64)
        Ud = Us[b].astype(np.float64)
        res = np.linalg.norm(Bs[b].astype(np.float64) - Ud.T @ (Ud @ X))
        bound = checks.RECON_PER_N * n * np.linalg.norm(Ud) ** 2 * np.linalg.norm(X)
        assert res <= bound, f"n={n} b={b}: residual {res:.3e} > {bound:.3e}"
        s = np.linalg.svd(Ud, compute_uv=False)
        err = np.abs(X - X_ref[b]).max() / np.abs(X_ref[b]).max()
        assert err <= 4 * n * U * (s[0] / s[-1]) ** 2
    pat = np.zeros(bbuf.size, dtype=bool)
    for b in range(batch):
        pat[b * strideB: b * strideB + n] = True
    assert np.array_equal(out.view(np.uint32)[~pat], bbuf.view(np.uint32)[~pat])


@pytest.mark.parametrize("n,nrhs", [(20, 3), (64, 9), (150, 4)])
def test_upper_sposv(n, nrhs):
    import torch

    import matrix_dense_linear_gb300 as bl
    batch = 6
    mats = _mats(n, batch, 1300 + n)
    mats[2] = synth.make_indefinite(mats[2], n // 2, delta=0.5)
    abuf = _pack_upper(mats, n, n, n * n)
    bbuf, Bs = _rhs(n, nrhs, batch, 1400 + n, n, n * nrhs)
    da = torch.from_numpy(abuf.copy()).cuda()
    db = torch.from_numpy(bbuf.copy()).cuda()
    info = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    assert bl.sposv_batched_uplo("U", da, n, n, n * n, db, nrhs, n, n * nrhs, batch, info) == 0
    torch.cuda.synchronize()
    inf = info.cpu().numpy()
    out = db.cpu().numpy()
    _check(abuf, da.cpu().numpy(), inf, n, n, n * n, batch, list(range(batch)), f"sposv U n={n}")
    assert inf[2] == n // 2 + 1
    for b in range(batch):
        X = _sol(out, n, nrhs, n, n * nrhs, b)
        if inf[b]:
            assert np.array_equal(X.view(np.uint32), Bs[b].view(np.uint32))
            continue
        A = checks.sym_from_lower(np.triu(np.asarray(mats[b]).astype(np.float32)).T)
        Xd = X.astype(np.float64)
        res = np.linalg.norm(Bs[b].astype(np.float64) - A @ Xd)
        assert res <= 2 * checks.RECON_PER_N * n * np.linalg.norm(A) * np.linalg.norm(Xd)
