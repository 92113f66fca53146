"""bl_spotrf_batched_static, the entry point that allocates nothing, through the
C-ABI (GPU).

It serves callers that cannot allocate device memory where they factor: a
library running inside a framework whose allocator it cannot reach, a
latency-bounded loop that cannot take the synchronization of cudaMalloc, a
process already at its memory limit. The scratch of the inverse-based panel
solve then comes from a fixed device array inside the library instead of a
caller workspace. Its results must agree with the call that takes a caller
workspace (bl_spotrf_batched_ws) within the tolerances of the parity tests,
on two calls in a row (the second call finds the first one's contents in the
shared array), and a call whose scratch would not fit must be rejected.

The file name puts it last in collection order: a run that stops at the first
failure has run every other test before this one. It builds what it needs, so
it also passes alone in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest

import synth
from tests import checks
from tests.gpu_helpers import assert_untouched

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20  # BL_SPOTRF_STATIC_SCRATCH_BYTES
INVERSE_BYTES = 128 * 128 * 4  # scratch per matrix of order > 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    from matrix_dense_linear_gb300 import build
    build.build()


def _batch(n, batch, seed):
    return synth.pack(lambda b: synth.gram(n, synth.rng(seed, b), "normal", float(n), 1.0),
                      n, batch, fill="nan")


def _static(bt):
    """Factor a copy of the batch through bl_spotrf_batched_static."""
    import torch

    import matrix_dense_linear_gb300 as bl
    A = torch.from_numpy(bt.buf.copy()).cuda()
    info = torch.full((bt.batch,), -7, dtype=torch.int32, device="cuda")
    code = bl.library().bl_spotrf_batched_static(A.data_ptr(), bt.n, bt.lda, bt.strideA,
                                                  bt.batch, info.data_ptr(),
                                                  torch.cuda.current_stream().cuda_stream)
    assert code == 0, f"bl_spotrf_batched_static returned {code}"
    torch.cuda.synchronize()
    return A.cpu().numpy(), info.cpu().numpy()


def _with_workspace(bt):
    """The same batch through bl_spotrf_batched_ws with a caller workspace."""
    import torch

    import matrix_dense_linear_gb300 as bl
    A = torch.from_numpy(bt.buf.copy()).cuda()
    info = torch.full((bt.batch,), -7, dtype=torch.int32, device="cuda")
    need = bl.workspace_bytes(bt.n, bt.batch)
    work = torch.empty(max(need // 4, 4), dtype=torch.float32, device="cuda")
    code = bl.library().bl_spotrf_batched_ws(A.data_ptr(), bt.n, bt.lda, bt.strideA, bt.batch,
                                              info.data_ptr(), work.data_ptr(), need,
                                              torch.cuda.current_stream().cuda_stream)
    assert code == 0, f"bl_spotrf_batched_ws returned {code}"
    torch.cuda.synchronize()
    return A.cpu().numpy(), info.cpu().numpy()


def _agree(bt, got, ref, what):
    (out_s, info_s), (out_w, info_w) = got, ref
    assert np.array_equal(info_s, info_w), what
    assert_untouched(out_s, bt.buf, bt, what=what)
    vs = synth.strided_view(out_s, bt.n, bt.lda, bt.strideA, bt.batch)
    vw = synth.strided_view(out_w, bt.n, bt.lda, bt.strideA, bt.batch)
    for b in range(bt.batch):
        Ls = np.tril(np.array(vs[b], dtype=np.float64))
        Lw = np.tril(np.array(vw[b], dtype=np.float64))
        e = checks.max_rel(Ls, Lw)
        assert e <= checks.MAXREL_PER_N * bt.n, f"{what} matrix {b}: max rel {e:.3e}"
        r = checks.recon_error(Ls, bt.lower(b))
        assert r <= checks.RECON_PER_N * bt.n, f"{what} matrix {b}: recon {r:.3e}"


def test_two_calls_in_a_row_match_the_workspace_call():
    # two different batches back to back: the second call reads the shared
    # array only where it has written it first
    first = _batch(512, 12, 1201)
    second = _batch(640, 9, 1202)
    for bt, what in ((first, "first call"), (second, "second call")):
        _agree(bt, _static(bt), _with_workspace(bt), what)


def test_orders_without_scratch():
    # n <= 128 needs no scratch; the call runs like bl_spotrf_batched
    bt = _batch(64, 300, 1203)
    _agree(bt, _static(bt), _with_workspace(bt), "n = 64")


def test_largest_batch_that_fits_and_the_first_that_does_not():
    import torch

    import matrix_dense_linear_gb300 as bl
    lib = bl.library()
    st = torch.cuda.current_stream().cuda_stream
    fit = STATIC_BYTES // INVERSE_BYTES  # 256 matrices of order > 128
    bt = _batch(256, fit, 1204)
    _agree(bt, _static(bt), _with_workspace(bt), f"batch {fit}")
    A = torch.zeros(256 * 256 * (fit + 1), device="cuda")
    info = torch.zeros(fit + 1, dtype=torch.int32, device="cuda")
    assert lib.bl_spotrf_batched_static(A.data_ptr(), 256, 256, 256 * 256, fit + 1,
                                         info.data_ptr(), st) == -10
    # the usual argument checks come first
    assert lib.bl_spotrf_batched_static(A.data_ptr(), -1, 256, 256 * 256, fit + 1,
                                         info.data_ptr(), st) == -2
    assert lib.bl_spotrf_batched_static(A.data_ptr(), 256, 255, 256 * 256, fit + 1,
                                         info.data_ptr(), st) == -3
    torch.cuda.synchronize()
