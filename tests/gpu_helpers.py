"""Run the CUDA path through the C-ABI on a synth.Batch and compare it with the
oracle (used by the -m gpu tests and nothing else)."""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

import oracle
import synth
from tests import checks


def run_gpu(bt: synth.Batch, route: int = 0, stream=None, info_fill: int = -7):
    """Copy the batch's whole buffer (with any leading offset) to the device,
    factor it in place through bl_spotrf_batched_ex, and bring it back.
    Returns (buffer after, info)."""
    import torch

    import matrix_dense_linear_gb300 as bl

    base = getattr(bt, "base", bt.buf)
    offset = (bt.buf.__array_interface__["data"][0] - base.__array_interface__["data"][0]) // 4
    dbuf = torch.from_numpy(base.copy()).cuda()
    info = torch.full((max(bt.batch, 1),), info_fill, dtype=torch.int32, device="cuda")
    ptr = dbuf.data_ptr() + 4 * offset
    code = bl.spotrf_batched_ex(ptr, bt.n, bt.lda, bt.strideA, bt.batch, info, stream, route)
    assert code == 0, f"bl_spotrf_batched_ex returned {code}"
    torch.cuda.synchronize()
    out = dbuf.cpu().numpy()[offset:offset + bt.buf.size]
    return out, info.cpu().numpy()[:bt.batch]


def slot_pattern(n: int, lda: int, strideA: int) -> np.ndarray:
    """Over one matrix's span: True where the element is not in the lower triangle."""
    span = max(strideA, lda * n)
    m = np.ones(span, dtype=bool)
    for j in range(n):
        m[j + j * lda: n + j * lda] = False
    return m


def assert_untouched(after: np.ndarray, before: np.ndarray, bt: synth.Batch, what=""):
    pat = slot_pattern(bt.n, bt.lda, bt.strideA)
    a32 = after.view(np.uint32)
    b32 = before.view(np.uint32)
    step = bt.strideA if bt.batch > 1 else pat.size
    for b in range(bt.batch):
        lo = b * step
        hi = min(lo + pat.size, a32.size)
        p = pat[:hi - lo]
        diff = np.count_nonzero(a32[lo:hi][p] != b32[lo:hi][p])
        assert diff == 0, f"{what}: matrix {b}: {diff} elements outside the lower triangle changed"
    # anything past the last slot (none with buffer_size) must be equal too
    tail = a32[(bt.batch - 1) * step + pat.size:] if bt.batch else a32
    assert np.array_equal(tail, b32[a32.size - tail.size:])


def compare(bt: synth.Batch, out: np.ndarray, info: np.ndarray,
            indices: Optional[Sequence[int]] = None, what: str = "") -> np.ndarray:
    """Oracle parity on the chosen matrices (all by default): info bit-exact, L
    within tolerance, reconstruction within budget. Returns the oracle's info."""
    idx = list(range(bt.batch)) if indices is None else list(indices)
    L_ref, info_ref, _ = oracle.potrf_batched(bt.buf, bt.n, bt.lda, bt.strideA, bt.batch,
                                              indices=idx)
    gv = synth.strided_view(out, bt.n, bt.lda, bt.strideA, bt.batch)
    av = bt.view()
    for t, b in enumerate(idx):
        checks.check_factor(np.array(gv[b]), L_ref[t], int(info[b]), int(info_ref[t]),
                            np.tril(np.array(av[b])), what=f"{what} matrix {b}")
    return info_ref
