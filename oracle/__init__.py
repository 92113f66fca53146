"""CPU oracle for batched SPOTRF and SPOTRS (column-major, strided batch, uplo
'L' or 'U').

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. The CUDA library never
links, loads or calls it, and it never calls the CUDA library.

The arithmetic lives in ``chol_ref.c`` (plain C, IEEE double, unblocked
Cholesky-Crout), ``dchol_ref.c`` (the same for a double-precision input) and
``potrs_ref.c`` (forward and backward substitution with the factor) and
``cchol_ref.c`` (the Hermitian factorization of a complex input); this
module only compiles them with gcc into
``oracle/_build/liboracle.so`` and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "chol_ref.c"), os.path.join(_HERE, "potrs_ref.c"),
         os.path.join(_HERE, "dchol_ref.c"), os.path.join(_HERE, "cchol_ref.c")]
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, no FMA contraction). Returns the .so path."""
    with _lock:
        if (not force and os.path.exists(_SO)
                and all(os.path.getmtime(_SO) >= os.path.getmtime(f) for f in _SRCS)):
            return _SO
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
               "-pthread", *_SRCS, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
        return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_potrf_one.restype = ctypes.c_int
        lib.oracle_potrf_one.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_int]
        lib.oracle_potrf_upper_one.restype = ctypes.c_int
        lib.oracle_potrf_upper_one.argtypes = lib.oracle_potrf_one.argtypes
        lib.oracle_potrf_batched_uplo.restype = ctypes.c_int
        lib.oracle_potrf_batched_uplo.argtypes = [
            ctypes.c_char, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
            ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_dpotrf_one.restype = ctypes.c_int
        lib.oracle_dpotrf_one.argtypes = lib.oracle_potrf_one.argtypes
        lib.oracle_dpotrf_upper_one.restype = ctypes.c_int
        lib.oracle_dpotrf_upper_one.argtypes = lib.oracle_potrf_one.argtypes
        lib.oracle_dpotrf_batched_uplo.restype = ctypes.c_int
        lib.oracle_dpotrf_batched_uplo.argtypes = lib.oracle_potrf_batched_uplo.argtypes
        lib.oracle_cpotrf_one.restype = ctypes.c_int
        lib.oracle_cpotrf_one.argtypes = lib.oracle_potrf_one.argtypes
        lib.oracle_cpotrf_upper_one.restype = ctypes.c_int
        lib.oracle_cpotrf_upper_one.argtypes = lib.oracle_potrf_one.argtypes
        lib.oracle_cpotrf_batched_uplo.restype = ctypes.c_int
        lib.oracle_cpotrf_batched_uplo.argtypes = lib.oracle_potrf_batched_uplo.argtypes
        lib.oracle_zpotrf_one.restype = ctypes.c_int
        lib.oracle_zpotrf_one.argtypes = lib.oracle_potrf_one.argtypes
        lib.oracle_zpotrf_upper_one.restype = ctypes.c_int
        lib.oracle_zpotrf_upper_one.argtypes = lib.oracle_potrf_one.argtypes
        lib.oracle_zpotrf_batched_uplo.restype = ctypes.c_int
        lib.oracle_zpotrf_batched_uplo.argtypes = lib.oracle_potrf_batched_uplo.argtypes
        lib.oracle_potrs_one.restype = None
        lib.oracle_potrs_one.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_int]
        lib.oracle_potrs_upper_one.restype = None
        lib.oracle_potrs_upper_one.argtypes = lib.oracle_potrs_one.argtypes
        lib.oracle_potrs_batched_uplo.restype = ctypes.c_int
        lib.oracle_potrs_batched_uplo.argtypes = [
            ctypes.c_char, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int]
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def _upper(uplo: str) -> bool:
    if uplo not in ("L", "U", "l", "u"):
        raise ValueError(f"uplo must be 'L' or 'U', not {uplo!r}")
    return uplo in ("U", "u")


def potrf_one(A: np.ndarray, uplo: str = "L") -> tuple[np.ndarray, int]:
    """Factor one dense matrix (only its lower triangle is used; with
    ``uplo="U"`` only its upper triangle).

    ``A`` is any n x n array; it is rounded to float32 first (the oracle's
    input type). Returns (the factor as float64 n x n, info): L[i, j] = l_ij
    (A = L L^T), or with "U" U[i, j] = u_ij (A = U^T U)."""
    a32 = np.asfortranarray(np.asarray(A, dtype=np.float32))
    n = a32.shape[0]
    L = np.zeros((n, n), dtype=np.float64, order="F")
    lib = _load()
    fn = lib.oracle_potrf_upper_one if _upper(uplo) else lib.oracle_potrf_one
    info = fn(a32.ctypes.data, n, max(1, n), L.ctypes.data, max(1, n))
    return np.ascontiguousarray(L), int(info)


def dpotrf_one(A: np.ndarray, uplo: str = "L") -> tuple[np.ndarray, int]:
    """Factor one double-precision matrix (``A`` is taken as float64, no
    rounding); otherwise as ``potrf_one``."""
    a64 = np.asfortranarray(np.asarray(A, dtype=np.float64))
    n = a64.shape[0]
    L = np.zeros((n, n), dtype=np.float64, order="F")
    lib = _load()
    fn = lib.oracle_dpotrf_upper_one if _upper(uplo) else lib.oracle_dpotrf_one
    info = fn(a64.ctypes.data, n, max(1, n), L.ctypes.data, max(1, n))
    return np.ascontiguousarray(L), int(info)


def dpotrf_batched(buf: np.ndarray, n: int, lda: int, strideA: int, batch: int,
                   indices: Optional[Sequence[int]] = None, nthreads: Optional[int] = None,
                   uplo: str = "L") -> tuple[np.ndarray, np.ndarray, int]:
    """``potrf_batched`` for a flat float64 batch."""
    lib = _load()
    buf = np.ascontiguousarray(buf, dtype=np.float64)
    if indices is None:
        src, sA, m = buf, strideA, batch
    else:
        idx = list(indices)
        m = len(idx)
        span = lda * n
        src = np.empty(max(1, m * span), dtype=np.float64)
        for t, b in enumerate(idx):
            src[t * span:(t + 1) * span] = buf[b * strideA: b * strideA + span]
        sA = span
    L = np.zeros((m, n, n), dtype=np.float64)
    info = np.zeros(m, dtype=np.int32)
    th = default_threads() if nthreads is None else nthreads
    used = lib.oracle_dpotrf_batched_uplo(b"U" if _upper(uplo) else b"L", src.ctypes.data, n,
                                          lda, sA, m, L.ctypes.data, n * n, info.ctypes.data,
                                          th)
    return L.transpose(0, 2, 1), info, int(used)


def cpotrf_one(A: np.ndarray, uplo: str = "L") -> tuple[np.ndarray, int]:
    """Factor one Hermitian matrix A = L L^H (``uplo="U"``: A = U^H U). ``A``
    is rounded to complex64 (the input type); only its lower (upper) triangle
    is read, and the diagonal's imaginary part is ignored. Returns (the factor
    as complex128 n x n, info)."""
    a64 = np.asfortranarray(np.asarray(A, dtype=np.complex64))
    n = a64.shape[0]
    L = np.zeros((n, n), dtype=np.complex128, order="F")
    lib = _load()
    fn = lib.oracle_cpotrf_upper_one if _upper(uplo) else lib.oracle_cpotrf_one
    info = fn(a64.ctypes.data, n, max(1, n), L.ctypes.data, max(1, n))
    return np.ascontiguousarray(L), int(info)


def zpotrf_one(A: np.ndarray, uplo: str = "L") -> tuple[np.ndarray, int]:
    """``cpotrf_one`` for a double-precision complex input (taken as
    complex128, no rounding)."""
    a = np.asfortranarray(np.asarray(A, dtype=np.complex128))
    n = a.shape[0]
    L = np.zeros((n, n), dtype=np.complex128, order="F")
    lib = _load()
    fn = lib.oracle_zpotrf_upper_one if _upper(uplo) else lib.oracle_zpotrf_one
    info = fn(a.ctypes.data, n, max(1, n), L.ctypes.data, max(1, n))
    return np.ascontiguousarray(L), int(info)


def cpotrf_batched(buf: np.ndarray, n: int, lda: int, strideA: int, batch: int,
                   indices: Optional[Sequence[int]] = None, nthreads: Optional[int] = None,
                   uplo: str = "L") -> tuple[np.ndarray, np.ndarray, int]:
    """``potrf_batched`` for a flat complex64 batch (element (i, j) of matrix b
    at ``buf[b*strideA + i + j*lda]``); a complex128 batch is factored by the
    double-precision-input form (ZPOTRF)."""
    lib = _load()
    dbl = np.asarray(buf).dtype == np.complex128
    buf = np.ascontiguousarray(buf, dtype=np.complex128 if dbl else np.complex64)
    if indices is None:
        src, sA, m = buf, strideA, batch
    else:
        idx = list(indices)
        m = len(idx)
        span = lda * n
        src = np.empty(max(1, m * span), dtype=buf.dtype)
        for t, b in enumerate(idx):
            src[t * span:(t + 1) * span] = buf[b * strideA: b * strideA + span]
        sA = span
    L = np.zeros((m, n, n), dtype=np.complex128)
    info = np.zeros(m, dtype=np.int32)
    th = default_threads() if nthreads is None else nthreads
    fn = lib.oracle_zpotrf_batched_uplo if dbl else lib.oracle_cpotrf_batched_uplo
    used = fn(b"U" if _upper(uplo) else b"L", src.ctypes.data, n,
                                          lda, sA, m, L.ctypes.data, n * n, info.ctypes.data,
                                          th)
    return L.transpose(0, 2, 1), info, int(used)


def potrf_batched(buf: np.ndarray, n: int, lda: int, strideA: int, batch: int,
                  indices: Optional[Sequence[int]] = None,
                  nthreads: Optional[int] = None,
                  uplo: str = "L") -> tuple[np.ndarray, np.ndarray, int]:
    """Factor matrices of a strided float32 batch.

    ``buf`` is flat float32 with A_b(i, j) at ``buf[b*strideA + i + j*lda]``.
    ``indices`` picks a subset of b (default: all). Returns (L, info, threads)
    with L[t, i, j] = l_ij of the t-th picked matrix (float64) and info[t];
    with ``uplo="U"`` the upper triangles are read and L[t, i, j] = u_ij.
    """
    lib = _load()
    buf = np.ascontiguousarray(buf, dtype=np.float32)
    if indices is None:
        src, sA, m = buf, strideA, batch
    else:
        idx = list(indices)
        m = len(idx)
        span = lda * n
        src = np.empty(max(1, m * span), dtype=np.float32)
        for t, b in enumerate(idx):
            src[t * span:(t + 1) * span] = buf[b * strideA: b * strideA + span]
        sA = span
    L = np.zeros((m, n, n), dtype=np.float64)  # [t, j, i]: column-major per matrix
    info = np.zeros(m, dtype=np.int32)
    th = default_threads() if nthreads is None else nthreads
    used = lib.oracle_potrf_batched_uplo(b"U" if _upper(uplo) else b"L", src.ctypes.data, n,
                                         lda, sA, m, L.ctypes.data, n * n, info.ctypes.data,
                                         th)
    return L.transpose(0, 2, 1), info, int(used)


def potrs_one(L: np.ndarray, B: np.ndarray, uplo: str = "L") -> np.ndarray:
    """Solve (L L^T) X = B for one factor (only its lower triangle is used);
    with ``uplo="U"`` solve (U^T U) X = B, U = ``L``'s upper triangle.

    ``L`` (n x n) and ``B`` (n x nrhs, or a vector) are rounded to float32
    first (the oracle's input type). Returns X as float64 of B's shape."""
    l32 = np.asfortranarray(np.asarray(L, dtype=np.float32))
    b = np.asarray(B, dtype=np.float32)
    vec = b.ndim == 1
    b32 = np.asfortranarray(b.reshape(b.shape[0], -1))
    n, nrhs = b32.shape
    X = np.zeros((n, nrhs), dtype=np.float64, order="F")
    lib = _load()
    fn = lib.oracle_potrs_upper_one if _upper(uplo) else lib.oracle_potrs_one
    fn(l32.ctypes.data, n, max(1, n), b32.ctypes.data, nrhs, max(1, n), X.ctypes.data,
       max(1, n))
    X = np.ascontiguousarray(X)
    return X[:, 0] if vec else X


def potrs_batched(lbuf: np.ndarray, n: int, lda: int, strideA: int, bbuf: np.ndarray,
                  nrhs: int, ldb: int, strideB: int, batch: int,
                  indices: Optional[Sequence[int]] = None,
                  nthreads: Optional[int] = None, uplo: str = "L") -> tuple[np.ndarray, int]:
    """Solve A_b X_b = B_b with the factors of a strided float32 batch.

    ``lbuf`` holds L_b(i, j) at ``lbuf[b*strideA + i + j*lda]`` (lower triangle
    read; with ``uplo="U"`` the upper factor U_b, upper triangle read),
    ``bbuf`` B_b(i, c) at ``bbuf[b*strideB + i + c*ldb]``. ``indices`` picks a
    subset of b. Returns (X, threads) with X[t, i, c] (float64)."""
    lib = _load()
    lbuf = np.ascontiguousarray(lbuf, dtype=np.float32)
    bbuf = np.ascontiguousarray(bbuf, dtype=np.float32)
    if indices is None:
        ls, sA, bs, sB, m = lbuf, strideA, bbuf, strideB, batch
    else:
        idx = list(indices)
        m = len(idx)
        spanL, spanB = lda * n, ldb * nrhs
        ls = np.empty(max(1, m * spanL), dtype=np.float32)
        bs = np.empty(max(1, m * spanB), dtype=np.float32)
        for t, b in enumerate(idx):
            ls[t * spanL:(t + 1) * spanL] = lbuf[b * strideA: b * strideA + spanL]
            bs[t * spanB:(t + 1) * spanB] = bbuf[b * strideB: b * strideB + spanB]
        sA, sB = spanL, spanB
    X = np.zeros((m, nrhs, n), dtype=np.float64)  # [t, c, i]: column-major per matrix
    th = default_threads() if nthreads is None else nthreads
    used = lib.oracle_potrs_batched_uplo(b"U" if _upper(uplo) else b"L", ls.ctypes.data, n,
                                         lda, sA, bs.ctypes.data, nrhs, ldb, sB, m,
                                         X.ctypes.data, n * nrhs, th)
    return X.transpose(0, 2, 1), int(used)
