"""The call with a workspace (bl_spotrf_batched_ws): the blocked route's panels
with at least two row blocks below the diagonal block are solved by the inverse
of that block (computed once per matrix and panel into the workspace, then one
tensor-core product per 128 rows). Parity against the oracle through the C-ABI,
in both storages, at the workloads' sizes and above, with poisoned memory
outside the triangles; failures, argument codes and the injected give-up."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests import checks
from tests.gpu_helpers import assert_untouched, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from matrix_dense_linear_gb300 import build
    build.build()


def _gram_batch(n, batch, seed, fill="nan", lda=None, strideA=None):
    return synth.pack(lambda b: synth.gram(n, synth.rng(seed, b), "normal", float(n), 1.0),
                      n, batch, lda=lda, strideA=strideA, fill=fill)


def run_ws(bt, uplo="L", work="auto", stream=None):
    """Factor the batch's buffer on the device through bl_spotrf_batched_ws."""
    import torch

    import matrix_dense_linear_gb300 as bl
    dbuf = torch.from_numpy(bt.buf.copy()).cuda()
    info = torch.full((max(bt.batch, 1),), -7, dtype=torch.int32, device="cuda")
    if work == "auto":
        nbytes = bl.workspace_bytes(bt.n, bt.batch)
        work = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device="cuda")
    code = bl.spotrf_batched_ws(dbuf, bt.n, bt.lda, bt.strideA, bt.batch, info, work,
                                stream=stream, uplo=uplo)
    assert code == 0, f"bl_spotrf_batched_ws returned {code}"
    torch.cuda.synchronize()
    return dbuf.cpu().numpy(), info.cpu().numpy()[:bt.batch]


@pytest.mark.parametrize("n", [384, 500, 512, 640, 1000, 1024])
def test_ws_parity_lower(n):
    bt = _gram_batch(n, 3, 900 + n, fill="nan" if n % 2 else "big")
    out, info = run_ws(bt)
    compare(bt, out, info, what=f"ws n={n}")
    assert_untouched(out, bt.buf, bt, what=f"ws n={n}")


@pytest.mark.parametrize("n", [384, 512, 1000])
def test_ws_parity_upper(n):
    """The upper storage holds the same symmetric matrix transposed: U = L^T of
    the lower oracle's factor; the strict lower triangle stays untouched."""
    batch = 2
    mats = [synth.gram(n, synth.rng(950 + n, b), "normal", float(n), 1.0) for b in range(batch)]
    low = synth.pack(lambda b: mats[b], n, batch, fill="nan")
    buf = np.full(batch * n * n, np.nan, dtype=np.float32)
    for b, M in enumerate(mats):
        for j in range(n):  # column j, rows 0..j: the upper triangle
            buf[b * n * n + j * n: b * n * n + j * n + j + 1] = M[: j + 1, j].astype(np.float32)
    up = synth.Batch(buf, n, n, n * n, batch, "nan")
    out, info = run_ws(up, uplo="U")
    assert not info.any()
    L_ref, info_ref, _ = oracle.potrf_batched(low.buf, n, n, n * n, batch)
    assert not info_ref.any()
    strict_low = np.tril(np.ones((n, n), dtype=bool), -1)
    for b in range(batch):
        G = out[b * n * n:(b + 1) * n * n].reshape(n, n).T  # G[i, j] = A_b(i, j)
        U = np.triu(G.astype(np.float64))
        checks.check_factor(U.T, L_ref[b], 0, 0, np.tril(np.array(low.view()[b])),
                            what=f"ws upper n={n} matrix {b}")
        assert np.isnan(G[strict_low]).all(), "strict lower triangle written"


def test_ws_without_workspace_is_the_plain_call():
    import matrix_dense_linear_gb300 as bl
    import torch
    n, batch = 512, 4
    bt = _gram_batch(n, batch, 960)
    out_ws, info_ws = run_ws(bt, work=None)
    dbuf = torch.from_numpy(bt.buf.copy()).cuda()
    info = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    assert bl.spotrf_batched(dbuf, n, n, n * n, batch, info) == 0
    torch.cuda.synchronize()
    assert np.array_equal(out_ws.view(np.uint32), dbuf.cpu().numpy().view(np.uint32))
    assert np.array_equal(info_ws, info.cpu().numpy())


def test_ws_workload_n1024_full_size():
    """The n = 1024 workload (512 matrices, the benchmark's shape) through the
    workspace call: 130 seeded matrices against the oracle, everything outside
    the lower triangles bitwise unchanged."""
    w = synth.WORKLOADS["n1024"]
    bt = synth.workload_batch("n1024", fill="nan")
    out, info = run_ws(bt)
    g = np.random.default_rng(w.wid)
    idx = sorted({0, bt.batch - 1, *g.choice(bt.batch, 128, replace=False).tolist()})
    info_ref = compare(bt, out, info, indices=idx, what="ws n1024")
    assert not info.any() and not info_ref.any()
    assert_untouched(out, bt.buf, bt, what="ws n1024")


def test_ws_large_order():
    """n = 2048 (16 panels, the inverse path on 14 of them): the leading 1024 x
    1024 block against the oracle and the whole reconstruction within budget."""
    n = 2048
    bt = _gram_batch(n, 1, 970)
    out, info = run_ws(bt)
    assert info[0] == 0
    assert_untouched(out, bt.buf, bt, what="ws n=2048")
    A_low = np.tril(np.array(bt.view()[0]))
    L = np.tril(np.array(synth.strided_view(out, n, n, n * n, 1)[0], dtype=np.float64))
    m = 1024
    L_ref, info_ref = oracle.potrf_one(checks.sym_from_lower(A_low[:m, :m]))
    assert info_ref == 0
    err = np.abs(L[:m, :m] - L_ref).max() / np.abs(L_ref).max()
    assert err <= checks.MAXREL_PER_N * m, f"leading block max rel {err:.3e}"
    rec = checks.recon_error(L, A_low)
    assert rec <= checks.RECON_PER_N * n, f"reconstruction {rec:.3e}"


@pytest.mark.parametrize("n", [512, 700])
def test_ws_info_cases(n):
    """Indefinite at seeded pivots in every panel, a NaN, a zero matrix, mixed
    with SPD matrices: info bit-exact, the leading block before the failure."""
    ks = [0, 130, n // 2, n - 1]
    mats = []
    for t in range(8):
        A = synth.gram(n, synth.rng(980 + n, t), "normal", float(n), 1.0)
        if t < len(ks):
            A = synth.make_indefinite(A, ks[t], delta=0.5)
        elif t == 4:
            A[n // 3, n // 4] = np.nan
            A[n // 4, n // 3] = np.nan
        elif t == 5:
            A[:] = 0.0
        mats.append(A)
    bt = synth.pack(lambda b: mats[b], n, len(mats), fill="nan")
    out, info = run_ws(bt)
    info_ref = compare(bt, out, info, what=f"ws info n={n}")
    assert list(info_ref[:4]) == [k + 1 for k in ks]
    assert_untouched(out, bt.buf, bt, what=f"ws info n={n}")


def test_ws_argument_codes():
    import matrix_dense_linear_gb300 as bl
    import torch
    n, batch = 512, 2
    A = torch.zeros(n * n * batch, device="cuda")
    info = torch.zeros(batch, dtype=torch.int32, device="cuda")
    need = bl.workspace_bytes(n, batch)
    work = torch.empty(need // 4 + 8, device="cuda")
    lib = bl.library()
    st = torch.cuda.current_stream().cuda_stream
    # misaligned workspace, too small a workspace; the uplo form shifts by one
    assert lib.bl_spotrf_batched_ws(A.data_ptr(), n, n, n * n, batch, info.data_ptr(),
                                    work.data_ptr() + 4, need, st) == -8
    assert lib.bl_spotrf_batched_ws(A.data_ptr(), n, n, n * n, batch, info.data_ptr(),
                                    work.data_ptr(), need - 1, st) == -9
    assert lib.bl_spotrf_batched_uplo_ws(b"U", A.data_ptr(), n, n, n * n, batch,
                                         info.data_ptr(), work.data_ptr(), need - 1, st) == -10
    assert lib.bl_spotrf_batched_uplo_ws(b"X", A.data_ptr(), n, n, n * n, batch,
                                         info.data_ptr(), work.data_ptr(), need, st) == -1
    # the usual checks come first
    assert lib.bl_spotrf_batched_ws(A.data_ptr(), -1, n, n * n, batch, info.data_ptr(),
                                    work.data_ptr() + 4, need, st) == -2
    torch.cuda.synchronize()


def test_ws_injected_timeout():
    """Class 5: the tensor-core product of the inverse-based panel solve gives up
    at its first bounded wait for every third matrix: those report -1, the others
    match the oracle, nothing outside the triangles changes, and the next call
    factors the whole batch."""
    import matrix_dense_linear_gb300 as bl
    lib = bl.library()
    n, batch = 512, 6
    bt = _gram_batch(n, batch, 990)
    assert lib.bl_debug_fail_first_wait(5, 3) == 0
    try:
        out, info = run_ws(bt)
    finally:
        assert lib.bl_debug_fail_first_wait(5, 0) == 0
    hit = [b for b in range(batch) if b % 3 == 0]
    rest = [b for b in range(batch) if b % 3 != 0]
    assert all(info[b] == -1 for b in hit), list(info)
    assert not info[rest].any(), list(info)
    compare(bt, out, info, indices=rest, what="ws give-up untouched matrices")
    assert_untouched(out, bt.buf, bt, what="ws after give-up")
    out2, info2 = run_ws(bt)
    compare(bt, out2, info2, what="ws after reset")
