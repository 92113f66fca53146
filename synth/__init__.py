"""Seeded synthetic inputs for batched single-precision Cholesky (SPOTRF, lower).

This module makes matrices and lays them out in memory. It holds none of the
factorization's arithmetic: no pivot, square root, substitution or trailing
update is computed here. Both the CPU oracle's tests and the CUDA path's tests
and benchmark draw their inputs from it, and from nothing else.

Layout (column-major, strided batch): element (i, j) of matrix b lives at
``buf[b * strideA + i + j * lda]``. Everything that is not the lower triangle of
a matrix (the strict upper triangle, the padding rows ``n .. lda-1`` of every
column, the gap between one matrix and the next) is filled with a chosen value:

* ``"mirror"`` writes the upper triangle as the transpose of the rounded lower
  triangle (what a user would pass), and ``pad_value`` everywhere else;
* ``"nan"`` / ``"big"`` poison everything outside the lower triangles with NaN
  or 1e30, so a test can prove that memory was neither read into the result nor
  written.

Randomness is counter based: matrix ``b`` of workload ``w`` is drawn from a
Philox generator keyed by ``(w, b)``, so any single matrix can be regenerated
alone and the same matrix comes out at any batch size or position.

Workloads (the five configurations of batched SPOTRF this library is measured
on; every matrix is formed in float64 and rounded once to float32):

* ``n32``   n=32,   batch=1024 (+16 indefinite), A = G G^T/32 + I,    G iid N(0,1)
* ``n64``   n=64,   batch=1024, A = G G^T/64 + 0.1 I,                 G iid N(0,1)
* ``n128``  n=128,  batch=1024, A = Q diag(lam) Q^T, Q from the QR of an iid
  N(0,1) matrix, lam iid log-uniform on [1e-3, 1]
* ``n256``  n=256,  batch=4096, A = G G^T/256 + I,                    G iid U(-1,1)
* ``n1024`` n=1024, batch=512,  A = G G^T/1024 + 1e-2 I,              G iid N(0,1)
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Optional

import numpy as np

F32 = np.float32
POISON = {"nan": np.float32(np.nan), "big": np.float32(1e30)}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int            # Philox key word 0
    n: int
    batch: int
    kind: str           # "gram-normal", "gram-uniform", "spectral"
    scale: float = 1.0  # A = G G^T / scale + shift I
    shift: float = 0.0
    extra_info: int = 0  # indefinite matrices appended after the SPD batch

    @property
    def lda(self) -> int:
        return self.n

    @property
    def strideA(self) -> int:
        return self.n * self.n


WORKLOADS = {
    "n32": Workload("n32", 1, 32, 1024, "gram-normal", 32.0, 1.0, extra_info=16),
    "n64": Workload("n64", 2, 64, 1024, "gram-normal", 64.0, 0.1),
    "n128": Workload("n128", 3, 128, 1024, "spectral"),
    "n256": Workload("n256", 4, 256, 4096, "gram-uniform", 256.0, 1.0),
    "n1024": Workload("n1024", 5, 1024, 512, "gram-normal", 1024.0, 1e-2),
}

# Margin of the indefinite matrices: the failing pivot is -INFO_DELTA.
INFO_DELTA = 0.5


def rng(wid: int, b: int, stream: int = 0) -> np.random.Generator:
    """Counter-based generator for matrix ``b`` of workload ``wid``."""
    key = np.array([(wid << 8) | stream, b], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def gram(n: int, g: np.random.Generator, dist: str, scale: float, shift: float) -> np.ndarray:
    """A = G G^T / scale + shift I in float64 (G n x n, iid normal or uniform)."""
    if dist == "normal":
        G = g.standard_normal((n, n))
    elif dist == "uniform":
        G = g.uniform(-1.0, 1.0, (n, n))
    else:
        raise ValueError(dist)
    A = (G @ G.T) / scale
    A[np.diag_indices(n)] += shift
    return 0.5 * (A + A.T)


def spectral(n: int, g: np.random.Generator, lo: float = 1e-3, hi: float = 1.0) -> np.ndarray:
    """A = Q diag(lam) Q^T, Q orthogonal from Householder QR of an iid N(0,1) matrix,
    lam iid log-uniform on [lo, hi]."""
    Q, _ = np.linalg.qr(g.standard_normal((n, n)))
    lam = np.exp(g.uniform(np.log(lo), np.log(hi), n))
    A = (Q * lam) @ Q.T
    return 0.5 * (A + A.T)


def spd_matrix(w: Workload, b: int) -> np.ndarray:
    """The float64 SPD matrix ``b`` of workload ``w`` (before rounding)."""
    g = rng(w.wid, b)
    if w.kind == "gram-normal":
        return gram(w.n, g, "normal", w.scale, w.shift)
    if w.kind == "gram-uniform":
        return gram(w.n, g, "uniform", w.scale, w.shift)
    if w.kind == "spectral":
        return spectral(w.n, g)
    raise ValueError(w.kind)


def info_pivot(w: Workload, t: int) -> int:
    """0-based pivot index that the t-th indefinite matrix fails at: the first
    two are the first and the last pivot, the rest are drawn."""
    if t == 0:
        return 0
    if t == 1:
        return w.n - 1
    return int(rng(w.wid, t, stream=1).integers(0, w.n))


def make_indefinite(A: np.ndarray, k: int, delta: float = INFO_DELTA) -> np.ndarray:
    """Shift the diagonal entry k of the SPD matrix A down so that the Schur
    complement of the leading k x k block at (k, k) becomes -delta.

    The leading k x k block is untouched, so every earlier pivot stays positive.
    The Schur complement is found with a general (LU) solve, not a Cholesky
    step: q = a_k^T A_k^{-1} a_k and a_kk <- q - delta. After rounding to
    float32 the complement is re-checked in float64 to stay below -delta/2.
    """
    A = A.copy()
    if k > 0:
        a = A[:k, k]
        q = float(a @ np.linalg.solve(A[:k, :k], a))
    else:
        q = 0.0
    A[k, k] = q - delta
    A32 = A.astype(F32).astype(np.float64)
    if k > 0:
        a = A32[:k, k]
        q32 = float(a @ np.linalg.solve(A32[:k, :k], a))
    else:
        q32 = 0.0
    assert A32[k, k] - q32 < -delta / 2, "indefinite matrix lost its margin"
    return A


def workload_matrix(w: Workload, b: int) -> np.ndarray:
    """Matrix b of the workload: SPD for b < w.batch, indefinite after."""
    if b < w.batch:
        return spd_matrix(w, b)
    t = b - w.batch
    assert t < w.extra_info
    return make_indefinite(spd_matrix(w, b), info_pivot(w, t))


# ----------------------------------------------------------------------------
# Memory layout
# ----------------------------------------------------------------------------

def strided_view(buf: np.ndarray, n: int, lda: int, strideA: int, batch: int) -> np.ndarray:
    """View ``v`` with v[b, i, j] = A_b(i, j) over a flat float32 buffer."""
    it = buf.itemsize
    return np.lib.stride_tricks.as_strided(
        buf, shape=(batch, n, n), strides=(strideA * it, it, lda * it), writeable=True)


def buffer_size(n: int, lda: int, strideA: int, batch: int) -> int:
    """Floats spanned by the batch, through the last padding row of the last column."""
    if batch <= 0 or n <= 0:
        return 0
    return (batch - 1) * strideA + lda * n


@dataclasses.dataclass
class Batch:
    buf: np.ndarray     # flat float32
    n: int
    lda: int
    strideA: int
    batch: int
    fill: str

    def view(self) -> np.ndarray:
        return strided_view(self.buf, self.n, self.lda, self.strideA, self.batch)

    def lower(self, b: int) -> np.ndarray:
        """Lower triangle of matrix b as a dense float32 n x n (upper zero)."""
        return np.tril(np.array(self.view()[b]))

    def outside_mask(self) -> np.ndarray:
        """Boolean mask over ``buf``: True where the element is NOT in a lower triangle."""
        m = np.ones(self.buf.shape, dtype=bool)
        if self.n and self.batch:
            mv = strided_view(m, self.n, self.lda, self.strideA, self.batch)
            tri = np.tril(np.ones((self.n, self.n), dtype=bool))
            for b in range(self.batch):
                mv[b][tri] = False
        return m


def pack(mats: Callable[[int], np.ndarray] | np.ndarray, n: int, batch: int, *,
         lda: Optional[int] = None, strideA: Optional[int] = None,
         fill: str = "mirror", pad_value: float = 0.0, offset: int = 0,
         workers: Optional[int] = None) -> Batch:
    """Round each matrix once to float32 and lay the batch out column-major.

    ``mats`` is an array (batch, n, n) or a function b -> n x n float64 matrix.
    Only the lower triangle of each matrix is used; ``fill`` says what goes
    everywhere else (see the module docstring). ``offset`` floats of fill are
    put in front of matrix 0 (to misalign the base address). Matrices are made
    on ``workers`` threads (default: one per core); each writes its own slot.
    """
    import concurrent.futures as cf
    import os

    lda = n if lda is None else lda
    strideA = lda * n if strideA is None else strideA
    size = offset + buffer_size(n, lda, strideA, batch)
    if fill == "mirror":
        outside = np.float32(pad_value)
    else:
        outside = POISON[fill]
    buf = np.full(size, outside, dtype=F32)
    core = buf[offset:]
    v = strided_view(core, n, lda, strideA, batch)
    tri = np.tril(np.ones((n, n), dtype=bool))

    def one(b: int) -> None:
        m = mats(b) if callable(mats) else mats[b]
        m32 = np.asarray(m).astype(F32)
        if fill == "mirror":
            if not np.array_equal(m32, m32.T):
                low = np.where(tri, m32, F32(0))
                m32 = low + np.tril(low, -1).T
            v[b] = m32
        else:
            v[b] = np.where(tri, m32, outside)

    nw = workers if workers is not None else min(32, os.cpu_count() or 1)
    if nw <= 1 or batch < 4:
        for b in range(batch):
            one(b)
    else:
        with cf.ThreadPoolExecutor(max_workers=nw) as ex:
            list(ex.map(one, range(batch)))
    out = Batch(core, n, lda, strideA, batch, fill)
    out.base = buf  # type: ignore[attr-defined]
    return out


def workload_batch(name: str, fill: str = "mirror", batch: Optional[int] = None,
                   include_info: bool = True) -> Batch:
    """The named workload laid out with its own lda and strideA."""
    w = WORKLOADS[name]
    nb = w.batch if batch is None else batch
    total = nb + (w.extra_info if include_info and batch is None else 0)
    return pack(lambda b: workload_matrix(w, b), w.n, total,
                lda=w.lda, strideA=w.strideA, fill=fill)
