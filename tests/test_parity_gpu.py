"""Parity of the CUDA path with the CPU oracle, through the C-ABI (GPU).

info is compared bit-exactly, L within max|L - L_oracle|/max|L_oracle| <=
1e-5 n, the reconstruction within the printed budget 2.38e-6 n (Frobenius,
full symmetric A), and every element outside the lower triangles (poisoned
with NaN or 1e30) must come back bitwise unchanged.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests import checks
from tests.gpu_helpers import assert_untouched, compare, run_gpu

pytestmark = pytest.mark.gpu

WARP, CTA, BLOCKED, TMEM, LEFT = 1, 2, 3, 4, 5


def _routes(n):
    r = [0, BLOCKED]
    if n <= 64:
        r.append(WARP)
    if n <= 128:
        r += [CTA, TMEM]
    else:
        r.append(LEFT)
    return sorted(set(r))


def _gram_batch(n, batch, seed, fill="nan", lda=None, strideA=None, offset=0, shift=1.0):
    return synth.pack(lambda b: synth.gram(n, synth.rng(seed, b), "normal", float(n), shift),
                      n, batch, lda=lda, strideA=strideA, fill=fill, offset=offset)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from matrix_dense_linear_gb300 import build
    build.build()


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 9, 16, 17, 31, 32, 33, 63, 64, 65, 96, 127,
                               128, 129, 192, 255, 256, 257, 500, 512])
def test_orders_every_route(n):
    batch = 9 if n <= 128 else 3
    bt = _gram_batch(n, batch, 200 + n, fill="nan" if n % 2 else "big")
    for route in _routes(n):
        out, info = run_gpu(bt, route)
        compare(bt, out, info, what=f"n={n} route={route}")
        assert_untouched(out, bt.buf, bt, what=f"n={n} route={route}")


@pytest.mark.parametrize("route", [0, LEFT])
@pytest.mark.parametrize("n", [1000, 1024])
def test_large_orders(n, route):
    bt = _gram_batch(n, 2, 300 + n, fill="nan")
    out, info = run_gpu(bt, route)
    compare(bt, out, info, what=f"n={n} route={route}")
    assert_untouched(out, bt.buf, bt, what=f"n={n} route={route}")


@pytest.mark.parametrize("n", [2048, 3000, 4096])
def test_larger_orders(n):
    """Orders above the workloads' (the blocked route's 1025 .. 4096 range, one
    matrix): the leading 1024 x 1024 block of L against the oracle (the factor
    of a leading principal block is that block of the factor), info bit-exact,
    and the reconstruction of the whole matrix within the budget."""
    bt = _gram_batch(n, 1, 350 + n, fill="nan")
    out, info = run_gpu(bt)
    assert info[0] == 0
    assert_untouched(out, bt.buf, bt, what=f"n={n}")
    A_low = np.tril(np.array(bt.view()[0]))
    L = np.tril(np.array(synth.strided_view(out, n, n, n * n, 1)[0], dtype=np.float64))
    m = 1024
    L_ref, info_ref = oracle.potrf_one(checks.sym_from_lower(A_low[:m, :m]))
    assert info_ref == 0
    err = np.abs(L[:m, :m] - L_ref).max() / np.abs(L_ref).max()
    assert err <= checks.MAXREL_PER_N * m, f"n={n}: leading block max rel {err:.3e}"
    rec = checks.recon_error(L, A_low)
    assert rec <= checks.RECON_PER_N * n, f"n={n}: reconstruction {rec:.3e}"


@pytest.mark.parametrize("n", [5, 32, 48, 64, 128, 200])
@pytest.mark.parametrize("layout", ["lda+1", "lda+3", "offset", "odd-stride"])
def test_alignment_and_strides(n, layout):
    kw = {}
    if layout == "lda+1":
        kw = dict(lda=n + 1)
    elif layout == "lda+3":
        kw = dict(lda=n + 3, strideA=(n + 3) * n + 7)
    elif layout == "offset":
        kw = dict(offset=1)
    else:
        kw = dict(strideA=n * n + 1)
    bt = _gram_batch(n, 5, 400 + n, fill="nan", **kw)
    for route in _routes(n):
        out, info = run_gpu(bt, route)
        compare(bt, out, info, what=f"n={n} {layout} route={route}")
        assert_untouched(out, bt.buf, bt, what=f"n={n} {layout} route={route}")


@pytest.mark.parametrize("n", [4, 20, 32, 64, 128, 300])
def test_info_cases(n):
    """Indefinite at seeded pivots (behind a positive diagonal), a NaN entry, a
    zero matrix, a negative first pivot, mixed with SPD matrices."""
    g = np.random.default_rng(n)
    ks = [0, n - 1, n // 2, int(g.integers(0, n))]
    mats = []
    for t in range(12):
        A = synth.gram(n, synth.rng(500 + n, t), "normal", float(n), 1.0)
        if t < len(ks):
            A = synth.make_indefinite(A, ks[t], delta=0.5)
        elif t == 5:
            A[n // 3, n // 4] = np.nan
            A[n // 4, n // 3] = np.nan
        elif t == 6:
            A[:] = 0.0
        elif t == 7:
            A[0, 0] = -1.0
        mats.append(A)
    bt = synth.pack(lambda b: mats[b], n, len(mats), fill="nan")
    for route in _routes(n):
        out, info = run_gpu(bt, route)
        info_ref = compare(bt, out, info, what=f"n={n} route={route}")
        assert list(info_ref[:4]) == [k + 1 for k in ks]
        assert info_ref[6] == 1 and info_ref[7] == 1 and info_ref[5] > 0
        assert_untouched(out, bt.buf, bt, what=f"n={n} route={route}")


@pytest.mark.parametrize("n", [32, 64, 128, 256])
def test_batch_position_invariance_and_determinism(n):
    """Matrix b factored alone or at position b of a larger batch gives the same
    bits, and two runs give the same bits."""
    big = _gram_batch(n, 37 if n < 256 else 7, 600 + n, fill="big")
    out1, info1 = run_gpu(big)
    out2, info2 = run_gpu(big)
    assert np.array_equal(out1.view(np.uint32), out2.view(np.uint32))
    assert np.array_equal(info1, info2)
    gv = synth.strided_view(out1, n, n, n * n, big.batch)
    for b in (0, big.batch // 2, big.batch - 1):
        one = synth.pack(lambda _: np.array(big.view()[b], dtype=np.float64), n, 1, fill="big")
        o, i = run_gpu(one)
        assert i[0] == info1[b]
        assert np.array_equal(np.tril(o.reshape(n, n).T).view(np.uint32),
                              np.tril(np.array(gv[b])).view(np.uint32))


@pytest.mark.parametrize("n", [17, 32, 48, 64, 100, 128])
def test_routes_agree(n):
    bt = _gram_batch(n, 6, 700 + n, fill="nan")
    outs = [run_gpu(bt, r)[0] for r in _routes(n)]
    v = [synth.strided_view(o, n, n, n * n, 6) for o in outs]
    for b in range(6):
        ref = np.tril(np.array(v[0][b], dtype=np.float64))
        for other in v[1:]:
            got = np.tril(np.array(other[b], dtype=np.float64))
            assert np.abs(got - ref).max() <= 2e-5 * n * np.abs(ref).max()


def test_n64_small_and_large_batch_kernels_agree():
    """n = 33 .. 64 runs two warps per matrix in small batches and one warp in
    large ones; the same matrices factored both ways agree with each other and
    with the oracle."""
    n, big = 48, 2000
    bt = _gram_batch(n, big, 760, fill="nan")
    out_big, info_big = run_gpu(bt)
    small = synth.pack(lambda b: np.array(bt.view()[b], dtype=np.float64), n, 8, fill="nan")
    out_small, info_small = run_gpu(small)
    assert not info_big[:8].any() and not info_small.any()
    gv = synth.strided_view(out_big, n, n, n * n, big)
    sv = synth.strided_view(out_small, n, n, n * n, 8)
    for b in range(8):
        a, c = np.tril(np.array(gv[b], dtype=np.float64)), np.tril(np.array(sv[b], dtype=np.float64))
        assert np.abs(a - c).max() <= 2e-5 * n * np.abs(a).max()
    compare(small, out_small, info_small, what="n=48 small batch")
    compare(bt, out_big, info_big, indices=[0, 999, 1999], what="n=48 large batch")


@pytest.mark.parametrize("n,batch,chunks", [(48, 10, 3), (128, 7, 0), (200, 5, 2), (32, 40, 1)])
def test_host_buffer_call(n, batch, chunks):
    """bl_spotrf_batched_host: slices over two streams, host buffers in and out,
    gaps between matrices and the upper triangles come back unchanged."""
    import torch

    import matrix_dense_linear_gb300 as bl
    bt = _gram_batch(n, batch, 780 + n, fill="nan", strideA=n * n + 5)
    host = torch.from_numpy(bt.buf.copy()).pin_memory()
    info_h = torch.full((batch,), -7, dtype=torch.int32).pin_memory()
    bl.factor_host(host, n, bt.lda, bt.strideA, batch, info_h, chunks=chunks)
    out, info = host.numpy(), info_h.numpy()
    compare(bt, out, info, what=f"host n={n} chunks={chunks}")
    assert_untouched(out, bt.buf, bt, what=f"host n={n}")


@pytest.mark.parametrize("n,batch", [(20, 100), (64, 1000), (100, 30), (128, 40), (129, 9),
                                     (200, 30), (256, 64), (300, 7)])
def test_host_call_pinned_and_pageable_agree(n, batch):
    """Pinned host buffers of n <= 128 are factored in place by the kernel over
    the host link, larger ones through kernels that copy only the lower
    triangles in and out; pageable ones take the copy path. All give the bits
    of the device call."""
    import torch

    import matrix_dense_linear_gb300 as bl
    bt = _gram_batch(n, batch, 860 + n, fill="nan")
    dev = torch.from_numpy(bt.buf.copy()).cuda()
    info_d = torch.empty(batch, dtype=torch.int32, device="cuda")
    bl.factor(dev, n, bt.lda, bt.strideA, batch, info_d)
    want = dev.cpu().numpy()
    for pinned in (True, False):
        host = torch.from_numpy(bt.buf.copy())
        info_h = torch.full((batch,), -7, dtype=torch.int32)
        if pinned:
            host, info_h = host.pin_memory(), info_h.pin_memory()
        bl.factor_host(host, n, bt.lda, bt.strideA, batch, info_h)
        assert np.array_equal(info_h.numpy(), info_d.cpu().numpy()), pinned
        assert np.array_equal(host.numpy().view(np.uint32), want.view(np.uint32)), pinned
    compare(bt, want, info_d.cpu().numpy(), indices=list(range(min(batch, 40))),
            what=f"host n={n}")


@pytest.mark.parametrize("offset,chunks", [(0, 0), (1, 3), (3, 1)])
def test_host_call_triangle_copies(offset, chunks):
    """The triangle copies of the host-buffer call (n > 128, pinned buffers):
    a buffer starting off a 16-byte boundary (the scalar copy), gaps between
    the matrices and the upper triangles poisoned, several slices per stream:
    the factors and info are the device call's bits and nothing else changes."""
    import torch

    import matrix_dense_linear_gb300 as bl
    n, batch = 260, 11
    bt = _gram_batch(n, batch, 905 + offset, fill="nan", strideA=n * n + 7)
    base = torch.full((bt.buf.size + offset,), float("nan"), dtype=torch.float32).pin_memory()
    base[offset:] = torch.from_numpy(bt.buf)
    host = base[offset:]
    info_h = torch.full((batch,), -7, dtype=torch.int32).pin_memory()
    dev = torch.from_numpy(bt.buf.copy()).cuda()
    info_d = torch.empty(batch, dtype=torch.int32, device="cuda")
    bl.factor(dev, n, bt.lda, bt.strideA, batch, info_d)
    want = dev.cpu().numpy()
    bl.factor_host(host, n, bt.lda, bt.strideA, batch, info_h, chunks=chunks)
    assert np.array_equal(info_h.numpy(), info_d.cpu().numpy())
    assert np.array_equal(host.numpy().view(np.uint32), want.view(np.uint32))
    assert np.isnan(base[:offset].numpy()).all()
    assert_untouched(host.numpy(), bt.buf, bt, what=f"host triangles offset={offset}")


def test_fma_probe():
    """The probe's rates are positive and FP64 is far below FP32 on this GPU
    (and below the FP32 roofline's unit count times the clock)."""
    import torch

    import matrix_dense_linear_gb300 as bl
    f32, f64 = bl.fma_probe(32), bl.fma_probe(64)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 0 < f64 < f32 <= sms * 128 * 2 * 2.2e9 / 1e12
    out = torch.zeros(1, device="cuda")
    import ctypes
    v = ctypes.c_double(0.0)
    assert bl.library().bl_fma_probe(16, out.data_ptr(), ctypes.byref(v), None) == -1
    assert bl.library().bl_fma_probe(32, None, ctypes.byref(v), None) == -2


def test_n_zero_and_batch_zero():
    import torch

    import matrix_dense_linear_gb300 as bl
    info = torch.full((5,), 9, dtype=torch.int32, device="cuda")
    A = torch.zeros(4, device="cuda")
    assert bl.spotrf_batched(A, 0, 1, 0, 5, info) == 0
    torch.cuda.synchronize()
    assert info.cpu().tolist() == [0] * 5
    assert bl.spotrf_batched(A, 3, 3, 9, 0, info) == 0


def test_nondefault_stream():
    import torch
    bt = _gram_batch(64, 20, 800, fill="nan")
    s = torch.cuda.Stream()
    out, info = run_gpu(bt, 0, stream=s)
    compare(bt, out, info, what="stream")


@pytest.mark.parametrize("n,batch", [(32, 300), (64, 1000), (128, 50), (300, 6)])
def test_cuda_graph_capture_replays_the_same_bits(n, batch):
    """The call is stream-ordered and allocates nothing, so it can be captured
    into a CUDA graph; a replay gives the eager call's bits."""
    import torch

    import matrix_dense_linear_gb300 as bl
    bt = _gram_batch(n, batch, 820 + n, fill="nan")
    src = torch.from_numpy(bt.buf.copy()).cuda()
    eager, work = src.clone(), src.clone()
    info_e = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    info_g = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    bl.factor(eager, n, bt.lda, bt.strideA, batch, info_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bl.factor(work, n, bt.lda, bt.strideA, batch, info_g, stream=torch.cuda.current_stream())
    for _ in range(2):  # replays start from the pristine input
        work.copy_(src)
        info_g.fill_(-7)
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(info_e, info_g) and not info_e.any()
    assert torch.equal(eager.view(torch.int32), work.view(torch.int32))


def test_concurrent_calls_from_host_threads():
    """Reentrant and safe across streams: four host threads, each with its own
    stream and buffers, factor at the same time; every result equals the one
    factored alone."""
    import threading

    import torch

    import matrix_dense_linear_gb300 as bl
    cases = [(20, 500), (64, 700), (100, 40), (256, 5)]
    bts = [_gram_batch(n, b, 840 + n, fill="nan") for n, b in cases]
    srcs = [torch.from_numpy(bt.buf.copy()).cuda() for bt in bts]
    alone = []
    for bt, src in zip(bts, srcs):
        a = src.clone()
        info = torch.empty(bt.batch, dtype=torch.int32, device="cuda")
        bl.factor(a, bt.n, bt.lda, bt.strideA, bt.batch, info)
        alone.append((a, info))
    torch.cuda.synchronize()
    outs = [src.clone() for src in srcs]
    infos = [torch.full((bt.batch,), -7, dtype=torch.int32, device="cuda") for bt in bts]
    errors = []

    def work(t):
        try:
            st = torch.cuda.Stream()
            bt = bts[t]
            for _ in range(3):
                with torch.cuda.stream(st):
                    outs[t].copy_(srcs[t])
                    bl.factor(outs[t], bt.n, bt.lda, bt.strideA, bt.batch, infos[t], stream=st)
            st.synchronize()
        except Exception as e:  # noqa: BLE001
            errors.append(e)

    threads = [threading.Thread(target=work, args=(t,)) for t in range(len(bts))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for (a, info), o, i in zip(alone, outs, infos):
        assert torch.equal(info, i)
        assert torch.equal(a.view(torch.int32), o.view(torch.int32))


@pytest.mark.parametrize("route,n", [(1, 8), (1, 16), (1, 32), (1, 64), (2, 32), (2, 64),
                                     (2, 80), (2, 96), (2, 100), (2, 128), (3, 256), (4, 100),
                                     (4, 128)])
def test_kernels_use_no_local_memory(route, n):
    import matrix_dense_linear_gb300 as bl
    ki = bl.kernel_info(route, n)
    assert ki["local_bytes"] == 0, ki
    assert ki["regs"] > 0 and ki["threads"] > 0


# ---------------------------------------------------------------------------
# The five workloads at full size, in the launch configuration the benchmark
# times (the automatic route); poisoned outside the lower triangles.
# ---------------------------------------------------------------------------

# matrices compared with the oracle per workload: None = all of them; k = the
# first, the last and k more drawn without replacement by a generator seeded
# with the workload's id (n1024: 130 of 512, about 3 s of oracle time on 16
# host cores; every other workload in full)
SAMPLE = {"n32": None, "n64": None, "n128": None, "n256": None, "n1024": 128}


@pytest.mark.parametrize("name", ["n32", "n64", "n128", "n256", "n1024"])
def test_workload_full_size(name):
    w = synth.WORKLOADS[name]
    bt = synth.workload_batch(name, fill="nan")
    out, info = run_gpu(bt)
    k = SAMPLE[name]
    if k is None:
        idx = None
    else:
        g = np.random.default_rng(w.wid)
        idx = sorted({0, bt.batch - 1, *g.choice(bt.batch, k, replace=False).tolist()})
    info_ref = compare(bt, out, info, indices=idx, what=name)
    if name == "n32":
        # the 16 indefinite matrices after the SPD batch
        exp = [synth.info_pivot(w, t) + 1 for t in range(w.extra_info)]
        assert list(info[w.batch:]) == exp
        assert not info[:w.batch].any()
    else:
        assert not info.any() and not info_ref.any()
    assert_untouched(out, bt.buf, bt, what=name)
