"""Failure reporting on the GPU, through the C-ABI.

1. A positive pivot below FLT_MIN (a subnormal) is a zero pivot in single
   precision: every single-precision route reports it in info, so a matrix
   with info = 0 never carries the infinite root such a pivot would give. The
   double-precision oracle passes that pivot, so these cases check the
   library's documented reading directly (info = k + 1) and compare only the
   leading block before the pivot with the oracle.
2. The internal-error path (info = -1): bl_debug_fail_first_wait makes the
   blocks of chosen matrices report their first bounded wait as timed out.
   Those matrices must come back with info = -1, every other matrix of the
   same launch must match the oracle, nothing outside the lower triangles may
   change, and a following normal call must factor the whole batch. No wait is
   made to hang: the injected timeout returns at once, and the copies and
   tensor-core operations already issued drain under their normal bounded wait.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests import checks
from tests.gpu_helpers import assert_untouched, compare, run_gpu

pytestmark = pytest.mark.gpu

WARP, CTA, BLOCKED, TMEM = 1, 2, 3, 4
SUBNORMAL = float(np.float32(1e-40))  # below FLT_MIN = 1.18e-38, exact in float32


@pytest.fixture(scope="module", autouse=True)
def _built():
    from matrix_dense_linear_gb300 import build
    build.build()


def _with_subnormal_pivot(n, seed, k):
    """SPD matrix whose row and column k are zero but for a_kk = SUBNORMAL:
    pivots 0..k-1 are those of the SPD matrix, pivot k is exactly SUBNORMAL."""
    A = synth.gram(n, synth.rng(seed, 0 if k is None else k + 1), "normal", float(n), 1.0)
    if k is not None:
        A[k, :] = 0.0
        A[:, k] = 0.0
        A[k, k] = SUBNORMAL
    return A


@pytest.mark.parametrize("route,n", [(WARP, 8), (WARP, 32), (WARP, 48), (WARP, 64),
                                     (CTA, 32), (CTA, 80), (CTA, 96), (CTA, 128),
                                     (BLOCKED, 200), (BLOCKED, 256), (TMEM, 128)])
def test_subnormal_pivot_fails(route, n):
    ks = sorted({0, n // 3, n - 1})
    mats = [_with_subnormal_pivot(n, 700 + n, k) for k in ks]
    mats.append(_with_subnormal_pivot(n, 700 + n, None))  # an SPD control
    bt = synth.pack(lambda b: mats[b], n, len(mats), fill="nan")
    out, info = run_gpu(bt, route)
    assert list(info) == [k + 1 for k in ks] + [0], (route, n, list(info))
    L_ref, info_ref, _ = oracle.potrf_batched(bt.buf, n, bt.lda, bt.strideA, bt.batch)
    # the double-precision oracle passes the subnormal pivot: the reading differs
    assert not info_ref.any()
    gv = synth.strided_view(out, n, bt.lda, bt.strideA, bt.batch)
    for t, k in enumerate(ks):
        if k > 0:
            L = np.tril(np.array(gv[t], dtype=np.float64))
            e = checks.max_rel(L[:k, :k], L_ref[t][:k, :k])
            assert e <= checks.MAXREL_PER_N * k, (route, n, k, e)
    checks.check_factor(np.array(gv[len(ks)]), L_ref[len(ks)], int(info[len(ks)]), 0,
                        bt.lower(len(ks)), what=f"route {route} n={n} control")
    assert_untouched(out, bt.buf, bt, what=f"route {route} n={n}")


def test_subnormal_pivot_fails_upper_and_complex():
    """The upper storage and the single-precision complex call read the same
    pivot the same way."""
    import torch

    import matrix_dense_linear_gb300 as bl
    for n in (24, 100, 256):
        k = n // 2
        A = _with_subnormal_pivot(n, 760 + n, k)
        # upper storage: column-major upper triangle = A's lower triangle transposed
        up = np.asfortranarray(np.triu(A.T)).astype(np.float32)
        dA = torch.from_numpy(up.ravel(order="F").copy()).cuda()
        info = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        bl.factor(dA, n, n, n * n, 1, info, uplo="U")
        torch.cuda.synchronize()
        assert int(info.item()) == k + 1, ("U", n, int(info.item()))
        # complex Hermitian (a real matrix through the complex call)
        C = np.asfortranarray(A.astype(np.complex64))
        dC = torch.from_numpy(C.ravel(order="F").copy()).cuda()
        info.fill_(-7)
        bl.factor_complex(dC, n, n, n * n, 1, info)
        torch.cuda.synchronize()
        assert int(info.item()) == k + 1, ("C", n, int(info.item()))


# ---------------------------------------------------------------------------
# The give-up path, by failure injection
# ---------------------------------------------------------------------------

# (kernel class, n, route, batch): the class's kernel runs on that route for
# every matrix of a 16-byte-aligned batch of that order
GIVE_UP_CASES = [
    (1, 128, CTA, 24),       # the block kernel's bulk-copy load, whole matrices
    (1, 256, BLOCKED, 12),   # the same kernel on the blocked route's diagonal blocks
    (2, 256, BLOCKED, 12),   # the tensor-core panel solve (with the fused update)
    (2, 512, BLOCKED, 6),    # the tensor-core panel solve, several row blocks a matrix
    (3, 512, BLOCKED, 6),    # the tensor-core trailing update
    (4, 128, TMEM, 24),      # the tensor-memory kernel
]
EVERY = 3


@pytest.mark.parametrize("klass,n,route,batch", GIVE_UP_CASES)
def test_injected_timeout_reports_minus_one(klass, n, route, batch):
    import matrix_dense_linear_gb300 as bl
    lib = bl.library()
    bt = synth.pack(lambda b: synth.gram(n, synth.rng(800 + n, b), "normal", float(n), 1.0),
                    n, batch, fill="nan")
    assert lib.bl_debug_fail_first_wait(klass, EVERY) == 0
    try:
        out, info = run_gpu(bt, route)
    finally:
        assert lib.bl_debug_fail_first_wait(klass, 0) == 0
    hit = [b for b in range(batch) if b % EVERY == 0]
    rest = [b for b in range(batch) if b % EVERY != 0]
    assert all(info[b] == -1 for b in hit), (klass, n, list(info))
    assert not info[rest].any(), (klass, n, list(info))
    # the matrices the injection did not touch are factored as usual
    compare(bt, out, info, indices=rest, what=f"class {klass} n={n} untouched matrices")
    assert_untouched(out, bt.buf, bt, what=f"class {klass} n={n} after give-up")
    # the library works normally afterwards, on the whole batch
    out2, info2 = run_gpu(bt, route)
    compare(bt, out2, info2, what=f"class {klass} n={n} after reset")
    assert_untouched(out2, bt.buf, bt, what=f"class {klass} n={n} after reset")


def test_injection_argument_checks():
    import matrix_dense_linear_gb300 as bl
    lib = bl.library()
    assert lib.bl_debug_fail_first_wait(0, 1) == -1
    assert lib.bl_debug_fail_first_wait(8, 1) == -1
    assert lib.bl_debug_fail_first_wait(1, -1) == -2
    for k in (1, 2, 3, 4, 5, 6, 7):
        assert lib.bl_debug_fail_first_wait(k, 0) == 0
