"""Batched single-precision Cholesky (SPOTRF, lower) on GB300: Python binding.

A thin ctypes layer over the C-ABI library ``libbl_spotrf.so`` (declared in
``include/bl_spotrf.h``). It only marshals arguments: every step of the
factorization runs in the library's CUDA kernels. PyTorch is used for device
memory and streams. If the library has not been built (see
``matrix_dense_linear_gb300.build``) every call raises; there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = ["ROUTE_AUTO", "ROUTE_WARP", "ROUTE_CTA", "ROUTE_BLOCKED", "ROUTE_TMEM", "ROUTE_LEFT", "MAX_N",
           "BLError",
           "library", "library_path", "spotrf_batched", "spotrf_batched_ex", "route",
           "kernel_info", "version", "factor", "factor_host", "spotrs_batched",
           "workspace_bytes", "spotrf_batched_ws",
           "sposv_batched", "solve", "factor_solve"]

ROUTE_AUTO, ROUTE_WARP, ROUTE_CTA, ROUTE_BLOCKED, ROUTE_TMEM, ROUTE_LEFT = 0, 1, 2, 3, 4, 5
MAX_N = 4096
_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libbl_spotrf.so")
_lib = None

# (name, restype, argtypes) of every symbol include/bl_spotrf.h declares
_VP, _I, _I64, _C = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_char
SYMBOLS = {
    "bl_spotrf_batched": (_I, [_VP, _I, _I, _I64, _I, _VP, _VP]),
    "bl_spotrf_batched_ex": (_I, [_VP, _I, _I, _I64, _I, _VP, _VP, _I]),
    "bl_spotrf_route": (_I, [_I, _I]),
    "bl_spotrf_kernel_info": (_I, [_I, _I, _VP, _VP, _VP, _VP, _VP]),
    "bl_spotrf_version": (ctypes.c_char_p, []),
    "bl_spotrf_batched_host": (_I, [_VP, _I, _I, _I64, _I, _VP, _VP, _VP, _I, _VP, _I]),
    "bl_spotrs_batched": (_I, [_VP, _I, _I, _I64, _VP, _I, _I, _I64, _I, _VP]),
    "bl_sposv_batched": (_I, [_VP, _I, _I, _I64, _VP, _I, _I, _I64, _I, _VP, _VP]),
    "bl_spotrf_batched_uplo": (_I, [_C, _VP, _I, _I, _I64, _I, _VP, _VP]),
    "bl_dpotrf_batched": (_I, [_VP, _I, _I, _I64, _I, _VP, _VP]),
    "bl_fma_probe": (_I, [_I, _VP, _VP, _VP]),
    "bl_cpotrf_batched": (_I, [_VP, _I, _I, _I64, _I, _VP, _VP]),
    "bl_cpotrf_batched_uplo": (_I, [_C, _VP, _I, _I, _I64, _I, _VP, _VP]),
    "bl_zpotrf_batched": (_I, [_VP, _I, _I, _I64, _I, _VP, _VP]),
    "bl_zpotrf_batched_uplo": (_I, [_C, _VP, _I, _I, _I64, _I, _VP, _VP]),
    "bl_dpotrf_batched_uplo": (_I, [_C, _VP, _I, _I, _I64, _I, _VP, _VP]),
    "bl_spotrf_batched_uplo_ex": (_I, [_C, _VP, _I, _I, _I64, _I, _VP, _VP, _I]),
    "bl_spotrs_batched_uplo": (_I, [_C, _VP, _I, _I, _I64, _VP, _I, _I, _I64, _I, _VP]),
    "bl_sposv_batched_uplo": (_I, [_C, _VP, _I, _I, _I64, _VP, _I, _I, _I64, _I, _VP, _VP]),
    "bl_debug_fail_first_wait": (_I, [_I, _I]),
    "bl_spotrf_workspace_bytes": (ctypes.c_size_t, [_I, _I]),
    "bl_spotrf_batched_ws": (_I, [_VP, _I, _I, _I64, _I, _VP, _VP, ctypes.c_size_t, _VP]),
    "bl_spotrf_batched_uplo_ws": (_I, [_C, _VP, _I, _I, _I64, _I, _VP, _VP, ctypes.c_size_t,
                                       _VP]),
    "bl_spotrf_batched_static": (_I, [_VP, _I, _I, _I64, _I, _VP, _VP]),
}


class BLError(RuntimeError):
    """A nonzero status from the library (negative: bad argument; positive: CUDA error)."""

    def __init__(self, code: int, what: str = ""):
        self.code = code
        kind = f"argument {-code} invalid" if code < 0 else f"cudaError_t {code}"
        super().__init__(f"bl_spotrf{(' ' + what) if what else ''}: status {code} ({kind})")


def library() -> ctypes.CDLL:
    """Load the C-ABI library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise ImportError(
                f"{library_path} is missing: build it with "
                "`python -m matrix_dense_linear_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(library_path)
        for name, (res, args) in SYMBOLS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def spotrf_batched(A, n: int, lda: int, strideA: int, batch: int, info, stream=None) -> int:
    """bl_spotrf_batched: A and info are device tensors (or raw device pointers).
    Returns the library status (0 = enqueued)."""
    return library().bl_spotrf_batched(_ptr(A), n, lda, strideA, batch, _ptr(info),
                                       _stream(stream))


def spotrf_batched_ex(A, n: int, lda: int, strideA: int, batch: int, info, stream=None,
                      route: int = ROUTE_AUTO) -> int:
    """bl_spotrf_batched_ex: as spotrf_batched with the kernel class forced."""
    return library().bl_spotrf_batched_ex(_ptr(A), n, lda, strideA, batch, _ptr(info),
                                          _stream(stream), route)


def _uplo(uplo) -> bytes:
    return uplo.encode() if isinstance(uplo, str) else bytes(uplo)


def spotrf_batched_uplo(uplo, A, n: int, lda: int, strideA: int, batch: int, info, stream=None,
                        route: int = ROUTE_AUTO) -> int:
    """bl_spotrf_batched_uplo(_ex): uplo "L" or "U" ("U": A = U^T U in the upper
    triangles; the lower triangle of a row-major matrix). Returns the status;
    argument indices count uplo as argument 1."""
    if route == ROUTE_AUTO:
        return library().bl_spotrf_batched_uplo(_uplo(uplo), _ptr(A), n, lda, strideA, batch,
                                                _ptr(info), _stream(stream))
    return library().bl_spotrf_batched_uplo_ex(_uplo(uplo), _ptr(A), n, lda, strideA, batch,
                                               _ptr(info), _stream(stream), route)


def spotrs_batched_uplo(uplo, L, n: int, lda: int, strideA: int, B, nrhs: int, ldb: int,
                        strideB: int, batch: int, stream=None) -> int:
    """bl_spotrs_batched_uplo: the solve with an upper ("U") or lower factor."""
    return library().bl_spotrs_batched_uplo(_uplo(uplo), _ptr(L), n, lda, strideA, _ptr(B),
                                            nrhs, ldb, strideB, batch, _stream(stream))


def sposv_batched_uplo(uplo, A, n: int, lda: int, strideA: int, B, nrhs: int, ldb: int,
                       strideB: int, batch: int, info, stream=None) -> int:
    """bl_sposv_batched_uplo: factor (upper or lower storage) and solve."""
    return library().bl_sposv_batched_uplo(_uplo(uplo), _ptr(A), n, lda, strideA, _ptr(B), nrhs,
                                           ldb, strideB, batch, _ptr(info), _stream(stream))


def dpotrf_batched(A, n: int, lda: int, strideA: int, batch: int, info, stream=None,
                   uplo="L") -> int:
    """bl_dpotrf_batched(_uplo): A is a float64 device tensor (or pointer)."""
    if uplo in ("L", b"L"):
        return library().bl_dpotrf_batched(_ptr(A), n, lda, strideA, batch, _ptr(info),
                                           _stream(stream))
    return library().bl_dpotrf_batched_uplo(_uplo(uplo), _ptr(A), n, lda, strideA, batch,
                                            _ptr(info), _stream(stream))


def cpotrf_batched(A, n: int, lda: int, strideA: int, batch: int, info, stream=None,
                   uplo="L", double: Optional[bool] = None) -> int:
    """bl_cpotrf_batched(_uplo), or bl_zpotrf_batched(_uplo) for a complex128
    tensor (or with double=True for a raw pointer): A is a complex device
    tensor (or pointer)."""
    if double is None:
        double = str(getattr(A, "dtype", "")) == "torch.complex128"
    lib = library()
    if uplo in ("L", b"L"):
        fn = lib.bl_zpotrf_batched if double else lib.bl_cpotrf_batched
        return fn(_ptr(A), n, lda, strideA, batch, _ptr(info), _stream(stream))
    fn = lib.bl_zpotrf_batched_uplo if double else lib.bl_cpotrf_batched_uplo
    return fn(_uplo(uplo), _ptr(A), n, lda, strideA, batch, _ptr(info), _stream(stream))


def factor_complex(A, n: int, lda: int, strideA: int, batch: int, info, stream=None,
                   uplo="L") -> None:
    """cpotrf_batched (complex64 or complex128), raising BLError on a nonzero status."""
    code = cpotrf_batched(A, n, lda, strideA, batch, info, stream, uplo)
    if code:
        raise BLError(code, "cpotrf")


def factor_double(A, n: int, lda: int, strideA: int, batch: int, info, stream=None,
                  uplo="L") -> None:
    """dpotrf_batched, raising BLError on a nonzero status."""
    code = dpotrf_batched(A, n, lda, strideA, batch, info, stream, uplo)
    if code:
        raise BLError(code, "dpotrf")


def fma_probe(precision: int = 32, stream=None) -> float:
    """bl_fma_probe: this device's FMA throughput in TFLOP/s (32 or 64 bit)."""
    import torch
    out = torch.zeros(1, dtype=torch.float64 if precision == 64 else torch.float32,
                      device="cuda")
    v = ctypes.c_double(0.0)
    code = library().bl_fma_probe(precision, _ptr(out), ctypes.byref(v), _stream(stream))
    if code:
        raise BLError(code, "fma_probe")
    return v.value


def route(n: int, batch: int) -> int:
    """bl_spotrf_route: the kernel class chosen for (n, batch); needs no GPU."""
    return library().bl_spotrf_route(n, batch)


def kernel_info(route_: int, n: int) -> dict:
    """bl_spotrf_kernel_info: registers, local bytes, shared bytes, threads."""
    vals = [ctypes.c_int(0) for _ in range(5)]
    code = library().bl_spotrf_kernel_info(route_, n, *[ctypes.byref(v) for v in vals])
    if code:
        raise BLError(code, "kernel_info")
    keys = ["regs", "local_bytes", "static_smem", "dynamic_smem", "threads"]
    return {k: v.value for k, v in zip(keys, vals)}


def spotrs_batched(L, n: int, lda: int, strideA: int, B, nrhs: int, ldb: int, strideB: int,
                   batch: int, stream=None) -> int:
    """bl_spotrs_batched: L and B are device tensors (or raw device pointers);
    X overwrites B. Returns the library status (0 = enqueued)."""
    return library().bl_spotrs_batched(_ptr(L), n, lda, strideA, _ptr(B), nrhs, ldb, strideB,
                                       batch, _stream(stream))


def sposv_batched(A, n: int, lda: int, strideA: int, B, nrhs: int, ldb: int, strideB: int,
                  batch: int, info, stream=None) -> int:
    """bl_sposv_batched: factor A in place, then solve into B where info == 0."""
    return library().bl_sposv_batched(_ptr(A), n, lda, strideA, _ptr(B), nrhs, ldb, strideB,
                                      batch, _ptr(info), _stream(stream))


def solve(L, n, lda, strideA, B, nrhs, ldb, strideB, batch, stream=None, uplo="L") -> None:
    """spotrs_batched(_uplo), raising BLError on a nonzero status."""
    if uplo in ("L", b"L"):
        code = spotrs_batched(L, n, lda, strideA, B, nrhs, ldb, strideB, batch, stream)
    else:
        code = spotrs_batched_uplo(uplo, L, n, lda, strideA, B, nrhs, ldb, strideB, batch,
                                   stream)
    if code:
        raise BLError(code, "spotrs")


def factor_solve(A, n, lda, strideA, B, nrhs, ldb, strideB, batch, info, stream=None,
                 uplo="L") -> None:
    """sposv_batched(_uplo), raising BLError on a nonzero status."""
    if uplo in ("L", b"L"):
        code = sposv_batched(A, n, lda, strideA, B, nrhs, ldb, strideB, batch, info, stream)
    else:
        code = sposv_batched_uplo(uplo, A, n, lda, strideA, B, nrhs, ldb, strideB, batch, info,
                                  stream)
    if code:
        raise BLError(code, "sposv")


def version() -> str:
    return library().bl_spotrf_version().decode()


def workspace_bytes(n: int, batch: int) -> int:
    """bl_spotrf_workspace_bytes: device bytes the workspace call can use."""
    return int(library().bl_spotrf_workspace_bytes(n, batch))


def spotrf_batched_ws(A, n: int, lda: int, strideA: int, batch: int, info, work,
                      work_bytes: Optional[int] = None, stream=None, uplo="L") -> int:
    """bl_spotrf_batched_ws / bl_spotrf_batched_uplo_ws: `work` is a device
    tensor (or pointer, or None); work_bytes defaults to the tensor's size."""
    if work_bytes is None:
        work_bytes = 0 if work is None or isinstance(work, int) else \
            int(work.numel() * work.element_size())
    if uplo in ("L", b"L"):
        return library().bl_spotrf_batched_ws(_ptr(A), n, lda, strideA, batch, _ptr(info),
                                              _ptr(work), work_bytes, _stream(stream))
    return library().bl_spotrf_batched_uplo_ws(_uplo(uplo), _ptr(A), n, lda, strideA, batch,
                                               _ptr(info), _ptr(work), work_bytes,
                                               _stream(stream))


def factor(A, n: int, lda: int, strideA: int, batch: int, info, stream=None,
           route_: int = ROUTE_AUTO, uplo="L", work=None) -> None:
    """Factor in place on the device; raises BLError on a nonzero status. With
    `work` (a device workspace of workspace_bytes(n, batch) bytes) the call is
    bl_spotrf_batched_ws (automatic route only)."""
    if work is not None:
        code = spotrf_batched_ws(A, n, lda, strideA, batch, info, work, stream=stream, uplo=uplo)
        if code:
            raise BLError(code)
        return
    if uplo in ("L", b"L"):
        code = spotrf_batched_ex(A, n, lda, strideA, batch, info, stream, route_)
    else:
        code = spotrf_batched_uplo(uplo, A, n, lda, strideA, batch, info, stream, route_)
    if code:
        raise BLError(code)


def factor_host(A_host, n: int, lda: int, strideA: int, batch: int, info_host,
                A_dev=None, info_dev=None, streams=None, chunks: int = 0,
                synchronize: bool = True) -> None:
    """Factor a batch that lives in (pinned) host memory through
    bl_spotrf_batched_host: slices of the batch go host -> device, are factored
    and come back, one stream per slice, so copies and factorization overlap.
    The device buffers are the caller's if given, else allocated by torch; the
    streams are the caller's (torch streams) or two made here (two slices
    measured best for the 16.8 MB n = 64 batch on GB300). The current stream
    waits for all of them; with `synchronize` the host waits too (else the
    results are on the host once the current stream's work is done)."""
    import torch
    if A_dev is None:
        A_dev = torch.empty_like(A_host, device="cuda")
    if info_dev is None:
        info_dev = torch.empty_like(info_host, device="cuda")
    cur = torch.cuda.current_stream()
    if streams is None:
        streams = [cur, torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(cur)  # the device buffers are free once earlier work is done
    arr = (ctypes.c_void_p * len(streams))(*[_stream(s) for s in streams])
    code = library().bl_spotrf_batched_host(_ptr(A_host), n, lda, strideA, batch,
                                            _ptr(info_host), _ptr(A_dev), _ptr(info_dev),
                                            chunks, arr, len(streams))
    if code:
        raise BLError(code, "host")
    for s in streams:
        cur.wait_stream(s)
    if synchronize:
        cur.synchronize()
