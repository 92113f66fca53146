#!/usr/bin/env python3
"""Benchmark of batched SPOTRF (lower, FP32, column-major) on GB300.

One step = one call of bl_spotrf_batched over one batch of a workload (every
kernel the route launches), on a replica that no earlier step touched since
the L2 was flushed. Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload n64] [--no-per-n] [--no-cpu-baseline]
  python bench.py --sweep     # batch sweep of the small orders, one JSON line per point
  python bench.py --op potrs --workload n256 --nrhs 16   # the solve with the factor

The headline workload is n=64, batch=1024 (A = G G^T/64 + 0.1 I); `per_n`
adds the same measurement for every workload (n = 32, 64, 128, 256, 1024).
Under torchrun (N > 1) every rank factors its own copy of the batch on its own
GPU (independent replicas, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batched SPOTRF matrices/s and GFLOP/s per n; achieved fraction of roofline"
UNIT = "matrices/s"
L2_FLUSH_BYTES = 512 << 20
REPLICA_CAP_BYTES = 96 << 30

# DRAM bytes (read + write) from one ncu pass over the workload's bench command
# (dram__bytes_read.sum + dram__bytes_write.sum, one-pass metrics), with the
# sha256 of the sources at capture time: a changed source reports null. Scope:
# one launch of the workload's one kernel (n <= 128), or one whole call, all
# its launches summed (the blocked route, whose `achieved` is per call too).
TRAFFIC = {
    # workload: (source files, sha256 prefix over them, bytes, scope)
    "n32": (('matrix_dense_linear_gb300/csrc/potrf_warp.cu', 'matrix_dense_linear_gb300/csrc/bl_common.cuh'), "67514fa4e72bb6b5", 4219904, "per launch"),
    "n64": (('matrix_dense_linear_gb300/csrc/potrf_warp.cu', 'matrix_dense_linear_gb300/csrc/bl_common.cuh'), "67514fa4e72bb6b5", 12660224, "per launch"),
    "n128": (('matrix_dense_linear_gb300/csrc/potrf_cta.cu', 'matrix_dense_linear_gb300/csrc/cta_common.cuh', 'matrix_dense_linear_gb300/csrc/bl_common.cuh', 'matrix_dense_linear_gb300/csrc/tc_sm100.cuh'), "7edaae49fb143436", 42140000, "per launch"),
    "n256": (('matrix_dense_linear_gb300/csrc/potrf_blocked.cu', 'matrix_dense_linear_gb300/csrc/potrf_cta.cu', 'matrix_dense_linear_gb300/csrc/cta_common.cuh', 'matrix_dense_linear_gb300/csrc/trsm_tc.cu', 'matrix_dense_linear_gb300/csrc/syrk_tc.cu', 'matrix_dense_linear_gb300/csrc/tc_sm100.cuh', 'matrix_dense_linear_gb300/csrc/bl_common.cuh'), "5039563aab3a57de", 1708000000, "per call (4 launches)"),
    "n1024": (('matrix_dense_linear_gb300/csrc/potrf_blocked.cu', 'matrix_dense_linear_gb300/csrc/potrf_cta.cu', 'matrix_dense_linear_gb300/csrc/cta_common.cuh', 'matrix_dense_linear_gb300/csrc/trsm_tc.cu', 'matrix_dense_linear_gb300/csrc/syrk_tc.cu', 'matrix_dense_linear_gb300/csrc/tc_sm100.cuh', 'matrix_dense_linear_gb300/csrc/bl_common.cuh'), "5039563aab3a57de", 6120000000, "per call (22 launches)"),
}


def peaks() -> dict:
    p = {"hbm_gbs": 6684.5, "sm_max_mhz": 2070.0, "source": "fallback"}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        p.update(hbm_gbs=float(m["hbm_gbs"]), sm_max_mhz=float(m["sm_max_mhz"]),
                 source="measured")
    except Exception:
        pass
    return p


def flops_per_matrix(n: int) -> float:
    return n ** 3 / 3.0


def alg_bytes_per_matrix(n: int) -> float:
    # lower triangle read + lower triangle written, fp32
    return 4.0 * n * (n + 1)


def sector_bytes_per_matrix(n: int) -> int:
    """The lower triangle in and out rounded to the 32-byte sectors DRAM moves,
    for columns that start on a sector (lda a multiple of 8 floats, as in every
    workload): column k's rows k..n-1 touch ceil(n/8) - floor(k/8) sectors, read
    once and written once (n = 32: 5120 bytes against 4224 algorithmic)."""
    return 2 * 32 * sum((n + 7) // 8 - k // 8 for k in range(n))


def launches_per_call(n: int, batch: int = 0) -> int:
    """Kernels one lower-storage call on a 16-byte-aligned batch launches: one
    for n <= 128; above, on large batches the left-looking order (per panel
    its update, factor and solve), else per 128-wide panel the diagonal factor,
    the panel solve and the trailing update, except that the last panel has
    only its factor and a one-tile trailing matrix is updated inside the panel
    solve when the call holds at most 2048 matrices and no delayed update is
    pending (the blocked driver's schedule)."""
    if n <= 128:
        return 1
    panels = (n + 127) // 128
    count, pending = 0, False
    sms = 152
    if n > 256 and batch * ((n - 1) // 128) >= 10 * sms:
        # the left-looking order of large batches: per panel its update by the
        # earlier panels (not the first), its diagonal factor, its panel solve
        # (not the last)
        return 3 * panels - 2
    for p in range(panels):
        count += 1  # diagonal factor
        m = n - 128 * (p + 1)
        if m <= 0:
            break
        fuse = not pending and m <= 128 and (m < 128 or batch <= 2048)
        count += 1  # panel solve
        if fuse:
            continue
        t = (m + 127) // 128
        if pending:
            pending = False
        elif m > 128 and batch * (t * (t + 1) // 2) >= 16 * sms:
            pending = True
        count += 1  # trailing update
    return count


def dominant_kernel(n: int) -> str:
    if n <= 32:
        return "potrf_warp_kernel"
    if n <= 64:
        return "potrf_warp64_kernel"
    if n <= 128:
        return "potrf_cta_kernel"
    return "syrk_tc_kernel"  # the trailing update of 16-byte aligned batches


def kernel_source(n: int) -> str:
    d = os.path.join(ROOT, "matrix_dense_linear_gb300", "csrc")
    if n <= 64:
        return os.path.join(d, "potrf_warp.cu")
    if n <= 128:
        return os.path.join(d, "potrf_cta.cu")
    return os.path.join(d, "syrk_tc.cu")


def traffic_for(name: str, n: int, batch: int | None = None):
    """The captured DRAM bytes of workload `name`, or None when its sources
    changed since the capture or the run's batch is not the workload's own
    (the figure was taken at that batch)."""
    ent = TRAFFIC.get(name)
    if not ent:
        return None
    import synth
    wl = synth.WORKLOADS.get(name)
    if wl is None or n != wl.n or (batch is not None and batch != wl.batch):
        return None
    srcs, sha, nbytes, _ = ent
    h = hashlib.sha256()
    for src in srcs:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    cur = h.hexdigest()
    return nbytes if cur.startswith(sha) else None


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.samples = []
        self.proc = None
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        win = [p for (t, p) in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in win:
            for nm, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        pw = [num(p[3]) for p in win if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(win),
                "power_w_max": max(pw) if pw else None}


def make_host_batch(name: str, batch: int | None = None):
    import synth
    return synth.workload_batch(name, fill="mirror", include_info=False, batch=batch)


class DeviceWorkload:
    """Pristine device copy + replicas + the L2 flush buffer for one workload."""

    def __init__(self, bt, steps: int, dev):
        import torch
        self.bt = bt
        self.dev = dev
        self.span = bt.buf.size
        self.nbytes = self.span * 4
        self.pristine = torch.from_numpy(bt.buf).to(dev)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        want = max(steps, -(-2 * l2 // max(self.nbytes, 1)))
        self.nrep = int(max(1, min(want, REPLICA_CAP_BYTES // max(self.nbytes, 1))))
        self.rep = torch.empty((self.nrep, self.span), dtype=torch.float32, device=dev)
        self.info = torch.zeros(bt.batch, dtype=torch.int32, device=dev)
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def refresh(self, k=None):
        rng = range(self.nrep) if k is None else [k]
        for i in rng:
            self.rep[i].copy_(self.pristine)

    def flush_l2(self):
        self.flush.fill_(1.0)

    uplo = "L"
    work = None  # a device workspace: the call is bl_spotrf_batched_ws
    route = 0    # a forced route (bl_spotrf_batched_ex / _uplo_ex), 0: the automatic one

    def use_workspace(self) -> None:
        import torch

        import matrix_dense_linear_gb300 as bl
        nbytes = bl.workspace_bytes(self.bt.n, self.bt.batch)
        self.work = torch.empty(max(nbytes // 4, 4), dtype=torch.float32, device=self.dev)

    def call(self, i: int, stream) -> None:
        import matrix_dense_linear_gb300 as bl
        bt = self.bt
        if self.route:
            code = bl.spotrf_batched_uplo(self.uplo, self.rep[i].data_ptr(), bt.n, bt.lda,
                                          bt.strideA, bt.batch, self.info, stream, self.route)
        elif self.work is not None:
            code = bl.spotrf_batched_ws(self.rep[i].data_ptr(), bt.n, bt.lda, bt.strideA,
                                        bt.batch, self.info, self.work, stream=stream,
                                        uplo=self.uplo)
        elif self.uplo == "L":
            code = bl.spotrf_batched(self.rep[i].data_ptr(), bt.n, bt.lda, bt.strideA, bt.batch,
                                     self.info, stream)
        else:
            code = bl.spotrf_batched_uplo(self.uplo, self.rep[i].data_ptr(), bt.n, bt.lda,
                                          bt.strideA, bt.batch, self.info, stream)
        if code:
            raise bl.BLError(code)


def time_steps(w: DeviceWorkload, steps: int, barrier, graph: bool = True) -> float:
    """Device time (ms) of exactly `steps` calls, each on a fresh replica; the
    replicas are refreshed and the L2 flushed outside the timed intervals.
    With `graph`, the calls of a chunk are captured once into a CUDA graph and
    the graph's replay is timed (device time without host launch overhead);
    otherwise the calls are launched one by one from Python."""
    import torch
    st = torch.cuda.current_stream()
    total = 0.0
    done = 0
    while done < steps:
        chunk = min(w.nrep, steps - done)
        g = None
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                cs = torch.cuda.current_stream().cuda_stream
                for i in range(chunk):
                    w.call(i, cs)
        w.refresh()
        w.flush_l2()
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        if g is not None:
            g.replay()
        else:
            for i in range(chunk):
                w.call(i, st.cuda_stream)
        e1.record(st)
        torch.cuda.synchronize()
        barrier()
        total += e0.elapsed_time(e1)
        done += chunk
        del g
    return total


def soak(w: DeviceWorkload, seconds: float) -> None:
    """Untimed calls for `seconds` (clock ramp and clock sampling under load)."""
    import torch
    st = torch.cuda.current_stream()
    t0 = time.time()
    i = 0
    while time.time() - t0 < seconds:
        k = i % w.nrep
        w.refresh(k)
        w.call(k, st.cuda_stream)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()


def e2e_steps(w: DeviceWorkload, steps: int, warmup: int, barrier) -> dict:
    """Same metric through the public host-buffer call (bl_spotrf_batched_host)
    on pinned host buffers, a fresh input each step. For n <= 128 the kernel
    reads the lower triangles from host memory and writes the factors back
    there (no staging copies); above, per slice (eight on two streams) a kernel
    copies the lower triangles to the device, the slice is factored and a
    kernel copies the factors and info back, so one slice's copy in overlaps
    another's factorization and copy back. Either way the bytes crossing the
    host link are the lower triangles and info."""
    import torch

    import matrix_dense_linear_gb300 as bl
    bt = w.bt
    host_in = torch.from_numpy(bt.buf).pin_memory()
    host = torch.empty_like(host_in).pin_memory()
    info_h = torch.zeros(bt.batch, dtype=torch.int32).pin_memory()
    A_dev = w.rep[0]
    st = torch.cuda.current_stream()
    streams = [st, torch.cuda.Stream()]
    for _ in range(warmup):
        host.copy_(host_in)
        bl.factor_host(host, bt.n, bt.lda, bt.strideA, bt.batch, info_h, A_dev, w.info, streams)
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        host.copy_(host_in)  # a fresh input each step, outside the timed interval
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        bl.factor_host(host, bt.n, bt.lda, bt.strideA, bt.batch, info_h, A_dev, w.info, streams,
                       synchronize=False)
        e1.record(st)  # after every stream's copies and kernels
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert not info_h.any().item(), "e2e run reported a failed factorization"
    # the median step (times the steps, the form the callers divide): the host
    # link is shared with the box's other work, and one slow step (measured
    # once: a whole run at 1.18 against 0.156 ms a step) would swamp a mean;
    # the mean and the slowest step are reported beside it
    total = statistics.median(times) * steps
    stats = {"mean_ms_per_step": sum(times) / steps, "max_ms_per_step": max(times),
             "statistic": "median of the steps"}
    tri = 4 * bt.n * (bt.n + 1) // 2 * bt.batch
    if bt.n <= 128:  # in place over the host link: the lower triangles each way
        return {"ms": total, "h2d": tri, "d2h": tri + 4 * bt.batch, **stats,
                "mode": "in place on pinned host memory over the host link (no staging copies)"}
    return {"ms": total, "h2d": tri, "d2h": tri + 4 * bt.batch, **stats,
            "mode": "per slice: lower triangles copied in by kernel, factor, factors and info "
                    "copied back by kernel; eight slices on two streams"}


def oracle_rate(bt, seconds: float = 3.0, max_matrices: int | None = None,
                nthreads: int | None = None) -> dict:
    """The CPU oracle, as it stands, on the host cores (all, or nthreads):
    matrices/s on a bounded sample (whole batch, or its first max_matrices),
    repeated >= `seconds`."""
    import oracle
    m = bt.batch if max_matrices is None else min(bt.batch, max_matrices)
    if nthreads == 1 and max_matrices is None:
        m = min(m, 256)  # a bounded single-core sample
    idx = None if m == bt.batch else list(range(m))
    th = oracle.default_threads() if nthreads is None else nthreads
    t0 = time.perf_counter()
    passes = 0
    while True:
        _, _, used = oracle.potrf_batched(bt.buf, bt.n, bt.lda, bt.strideA, bt.batch,
                                          indices=idx, nthreads=th)
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": passes * m / dt, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"{passes} pass(es) over {m} of {bt.batch} matrices (n={bt.n}), "
                      f"{dt:.1f} s on {used} host threads",
            "gflops": passes * m * flops_per_matrix(bt.n) / dt / 1e9}


def oracle_sample_size(n: int) -> int | None:
    # about a second or more of double-precision work per pass on 16 cores
    return {256: 512, 1024: 32}.get(n)


def roofline_entry(name: str, n: int, batch: int, ms_per_call: float, pk: dict, sms: int,
                   calls_per_launch_avg: float | None = None) -> dict:
    fp32_peak = sms * 128 * 2 * pk["sm_max_mhz"] * 1e6 / 1e12  # TFLOP/s
    t = ms_per_call / 1e3
    bytes_ = alg_bytes_per_matrix(n) * batch
    flops = flops_per_matrix(n) * batch
    t_hbm = bytes_ / (pk["hbm_gbs"] * 1e9)
    t_alu = flops / (fp32_peak * 1e12)
    if t_hbm >= t_alu:
        sec = sector_bytes_per_matrix(n) * batch
        return {"bound": "hbm", "achieved": bytes_ / t / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": (bytes_ / t / 1e9) / pk["hbm_gbs"],
                "roof_ms": t_hbm * 1e3,
                # the same against the sector-rounded bytes (the least DRAM can move)
                "sector_bytes_per_matrix": sector_bytes_per_matrix(n),
                "frac_sector_rounded": (sec / t / 1e9) / pk["hbm_gbs"]}
    return {"bound": "alu", "achieved": flops / t / 1e12, "peak": fp32_peak,
            "unit": "TFLOP/s", "frac": (flops / t / 1e12) / fp32_peak, "roof_ms": t_alu * 1e3}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest x over the ranks of the default process group (the slowest
    rank's time); x itself when running alone."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, batch: int, steps: int, ms: float) -> float:
    """Whole-job matrices/s: every rank factors `batch` matrices per step (weak
    scaling), timed as the max over ranks of `steps` steps."""
    return world * batch * steps / (ms / 1e3)


def run_ours(args, rank: int, world: int, barrier) -> dict | None:
    import torch

    import matrix_dense_linear_gb300 as bl
    bl.library()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pk = peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    import synth
    w_desc = synth.WORKLOADS[args.workload]

    bt = make_host_batch(args.workload, args.batch)
    w = DeviceWorkload(bt, args.steps, dev)
    for i in range(args.warmup):
        w.refresh(i % w.nrep)
        w.call(i % w.nrep, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()

    sampler = ClockSampler(dev.index).start() if rank == 0 else None
    t_s0 = time.time()
    soak(w, args.soak)
    ms = time_steps(w, args.steps, barrier)
    ms_direct = time_steps(w, args.steps, barrier, graph=False)
    soak(w, 0.5)
    t_s1 = time.time()
    if sampler:
        sampler.stop()
    ms = max_over_ranks(ms, world, dev)

    # check this run's output on its last replica (info only; parity is the tests')
    info = w.info.cpu().numpy()
    assert not info.any(), "benchmark factorization reported failures"

    lat_us = single_call_us(w) if rank == 0 else None
    e2e = e2e_steps(w, args.steps, min(args.warmup, 3), barrier)
    e2e["ms"] = max_over_ranks(e2e["ms"], world, dev)

    n, batch = bt.n, bt.batch
    per_call = ms / args.steps
    value = job_rate(world, batch, args.steps, ms)
    rf = roofline_entry(args.workload, n, batch, per_call, pk, sms)
    nl = launches_per_call(n, batch)
    roof = {"bound": rf["bound"], "achieved": rf["achieved"], "peak": rf["peak"],
            "unit": rf["unit"], "frac": rf["frac"], "traffic": traffic_for(args.workload, n, batch),
            "traffic_scope": TRAFFIC[args.workload][3] if args.workload in TRAFFIC else None,
            "kernel": dominant_kernel(n), "peak_source": pk["source"],
            "peak_note": ("HBM: measured copy bandwidth" if rf["bound"] == "hbm" else
                          f"FP32: {sms} SMs x 128 FMA x 2 x {pk['sm_max_mhz']:.0f} MHz")}
    for k in ("sector_bytes_per_matrix", "frac_sector_rounded"):
        if k in rf:
            roof[k] = rf[k]
    if nl > 1:
        roof["note"] = "multi-launch route: achieved is per call over all its launches"
    if rank != 0:
        return None

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_call, "higher_is_better": True,
        "ms_per_step_direct_launch": ms_direct / args.steps,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "gflops": value * flops_per_matrix(n) / 1e9,
        "config": {"workload": f"{args.workload}: n={n}, batch={batch}, lda={bt.lda}, "
                               f"strideA={bt.strideA}, {w_desc.kind} SPD",
                   "n": n, "batch": batch, "lda": bt.lda, "strideA": bt.strideA,
                   "route": bl.route(n, batch),
                   "l2": "flushed before each timed chunk; every step factors its own "
                         "replica, untouched since the flush",
                   "timing": "CUDA events around the replay of a CUDA graph of the K calls",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "e2e": {"value": job_rate(world, batch, args.steps, e2e["ms"]), "unit": UNIT,
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": e2e["ms"] / args.steps, "mode": e2e["mode"],
                "statistic": e2e["statistic"], "mean_ms_per_step": e2e["mean_ms_per_step"],
                "max_ms_per_step": e2e["max_ms_per_step"]},
        "gpu_launches": nl * args.steps,
        "single_call_us": lat_us,
        "clocks": sampler.summary(t_s0, t_s1) if sampler else None,
        "fma_probe_tflops": {"f32": bl.fma_probe(32), "f64": bl.fma_probe(64)},
    }
    if args.cpu_baseline and world == 1:
        out["cpu_baseline"] = oracle_rate(bt, 3.0, oracle_sample_size(n))
        one = oracle_rate(bt, 2.0, oracle_sample_size(n), nthreads=1)
        out["cpu_baseline"]["one_core"] = {"value": one["value"], "sample": one["sample"]}
    del w
    torch.cuda.empty_cache()

    if args.per_n:
        rows = []
        for name in ["n32", "n64", "n128", "n256", "n1024"]:
            if name == args.workload:
                rows.append({"workload": name, "n": n, "batch": batch,
                             "ms_per_call": per_call, "matrices_per_s": batch / (per_call / 1e3),
                             "gflops": batch * flops_per_matrix(n) / (per_call / 1e3) / 1e9,
                             "roofline": {**{k: rf[k] for k in ("bound", "frac", "roof_ms",
                                                                "frac_sector_rounded") if k in rf},
                                          "traffic": roof["traffic"],
                                          "traffic_scope": roof["traffic_scope"]},
                             "launches_per_call": nl, "e2e": out["e2e"],
                             "oracle_matrices_per_s": out.get("cpu_baseline", {}).get("value")})
                continue
            b2 = make_host_batch(name)
            w2 = DeviceWorkload(b2, args.steps, dev)
            for i in range(min(args.warmup, w2.nrep)):
                w2.refresh(i)
                w2.call(i, torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            ms2 = time_steps(w2, args.steps, lambda: None)
            assert not w2.info.cpu().numpy().any()
            pc = ms2 / args.steps
            r2 = roofline_entry(name, b2.n, b2.batch, pc, pk, sms)
            row = {"workload": name, "n": b2.n, "batch": b2.batch, "ms_per_call": pc,
                   "matrices_per_s": b2.batch / (pc / 1e3),
                   "gflops": b2.batch * flops_per_matrix(b2.n) / (pc / 1e3) / 1e9,
                   "roofline": {k: r2[k] for k in ("bound", "frac", "roof_ms",
                                                   "frac_sector_rounded") if k in r2},
                   "launches_per_call": launches_per_call(b2.n, b2.batch)}
            row["roofline"]["traffic"] = traffic_for(name, b2.n, b2.batch)
            row["roofline"]["traffic_scope"] = TRAFFIC[name][3] if name in TRAFFIC else None
            # the same workload end to end through the host-buffer call
            e2 = e2e_steps(w2, min(args.steps, 5), 2, lambda: None)
            row["e2e"] = {"value": b2.batch * min(args.steps, 5) / (e2["ms"] / 1e3),
                          "unit": UNIT, "ms_per_step": e2["ms"] / min(args.steps, 5),
                          "h2d_bytes_per_step": e2["h2d"], "d2h_bytes_per_step": e2["d2h"],
                          "mode": e2["mode"], "statistic": e2["statistic"],
                          "mean_ms_per_step": e2["mean_ms_per_step"]}
            if b2.n > 128:
                # the same workload through bl_spotrf_batched_ws (a caller-owned
                # workspace, allocated once outside the timed region)
                w2.use_workspace()
                for i in range(min(args.warmup, w2.nrep)):
                    w2.refresh(i)
                    w2.call(i, torch.cuda.current_stream().cuda_stream)
                torch.cuda.synchronize()
                ms3 = time_steps(w2, args.steps, lambda: None)
                assert not w2.info.cpu().numpy().any()
                pc3 = ms3 / args.steps
                r3 = roofline_entry(name, b2.n, b2.batch, pc3, pk, sms)
                row["workspace_call"] = {
                    "call": "bl_spotrf_batched_ws", "ms_per_call": pc3,
                    "matrices_per_s": b2.batch / (pc3 / 1e3),
                    "gflops": b2.batch * flops_per_matrix(b2.n) / (pc3 / 1e3) / 1e9,
                    "roofline": {k: r3[k] for k in ("bound", "frac", "roof_ms")},
                    "workspace_bytes": int(w2.work.numel() * 4)}
            if args.cpu_baseline:
                ob = oracle_rate(b2, 1.0, oracle_sample_size(b2.n))
                row["oracle_matrices_per_s"] = ob["value"]
                row["oracle_cores"] = ob["cores"]
            rows.append(row)
            del w2
            torch.cuda.empty_cache()
        out["per_n"] = rows
    return out


def single_call_us(w: DeviceWorkload, reps: int = 5) -> float:
    """Latency of one call launched from the host (median over reps): events
    around one launch on an idle stream, cold L2, replica untouched."""
    import torch
    st = torch.cuda.current_stream()
    ts = []
    for r in range(reps):
        k = r % w.nrep
        w.refresh(k)
        w.flush_l2()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        w.call(k, st.cuda_stream)
        e1.record(st)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts)


def run_sweep(args) -> list:
    """Batch sweep of the latency-scale orders (n = 32, 64, 128) up to 65536
    matrices: per point the median over 5 timed replays of K calls (graph,
    cold replicas), the single-call latency and the roofline fraction. Batches
    beyond a workload's own are the workload's matrices repeated."""
    import torch

    import matrix_dense_linear_gb300 as bl
    bl.library()
    dev = torch.device("cuda", 0)
    pk = peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rows = []
    for name in ("n32", "n64", "n128"):
        base = make_host_batch(name)
        for batch in (1, 16, 152, 1024, 4096, 16384, 65536):
            if name == "n128" and batch > 16384:
                continue
            reps = -(-batch // base.batch)
            buf = np.tile(base.buf[: base.batch * base.strideA], reps)[: batch * base.strideA]
            bt = type(base)(buf=np.ascontiguousarray(buf), n=base.n, lda=base.lda,
                            strideA=base.strideA, batch=batch, fill=base.fill)
            w = DeviceWorkload(bt, args.steps, dev)
            for i in range(min(args.warmup, w.nrep)):
                w.refresh(i)
                w.call(i, torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            k = min(args.steps, w.nrep)
            ms = statistics.median(time_steps(w, k, lambda: None) / k for _ in range(5))
            lat = single_call_us(w)
            assert not w.info.cpu().numpy().any()
            rf = roofline_entry(name, bt.n, batch, ms, pk, sms)
            row = {"sweep": name, "n": bt.n, "batch": batch, "ms_per_call": ms,
                   "single_call_us": lat, "matrices_per_s": batch / (ms / 1e3),
                   "roofline": {k2: rf[k2] for k2 in ("bound", "frac", "roof_ms")},
                   "calls_timed": k}
            print(json.dumps(row), flush=True)
            rows.append(row)
            del w
            torch.cuda.empty_cache()
    return rows


# (n, batch) pairs at which the pages quote their own timings (other hardware)
PAGES_SHAPES = "32x4096,64x1024,128x256,128x8192,256x64,512x16,512x640,1024x4,1024x60,17x16384"


def run_shapes(args) -> list:
    """Time arbitrary (n, batch) shapes, one JSON line each: A = G G^T / n + I
    (G iid normal, 64 distinct matrices repeated to fill the batch), packed
    lda = n, strideA = n^2; K calls per point on cold replicas (graph replay,
    L2 flushed before each replay), median over 3 replays."""
    import torch

    import matrix_dense_linear_gb300 as bl
    import synth
    bl.library()
    dev = torch.device("cuda", 0)
    pk = peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rows = []
    for spec in args.shapes.split(","):
        n, batch = (int(x) for x in spec.lower().split("x"))
        distinct = min(batch, 64)
        base = synth.pack(lambda b: synth.gram(n, synth.rng(6, b), "normal", float(n), 1.0),
                          n, distinct)
        reps = -(-batch // distinct)
        buf = np.ascontiguousarray(np.tile(base.buf, reps)[: batch * n * n])
        bt = type(base)(buf=buf, n=n, lda=n, strideA=n * n, batch=batch, fill=base.fill)
        w = DeviceWorkload(bt, args.steps, dev)
        w.uplo = args.uplo
        w.route = args.route
        if args.ws:
            w.use_workspace()
        for i in range(min(args.warmup, w.nrep)):
            w.refresh(i)
            w.call(i, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        k = min(args.steps, w.nrep)
        ms = statistics.median(time_steps(w, k, lambda: None) / k for _ in range(3))
        assert not w.info.cpu().numpy().any()
        rf = roofline_entry("shape", n, batch, ms, pk, sms)
        row = {"shape": spec, "uplo": args.uplo, "workspace": bool(args.ws), "route": args.route,
               "n": n,
               "batch": batch, "ms_per_call": ms,
               "us_per_call": ms * 1e3, "matrices_per_s": batch / (ms / 1e3),
               "tflops": flops_per_matrix(n) * batch / (ms / 1e3) / 1e12,
               "roofline": {k2: rf[k2] for k2 in ("bound", "frac", "roof_ms")},
               "calls_timed": k}
        print(json.dumps(row), flush=True)
        rows.append(row)
        del w
        torch.cuda.empty_cache()
    return rows


# FP64 peak of one GB300 when the probe cannot run: NVIDIA's nominal figure;
# the f64 rows use the library's FMA probe (bl_fma_probe) when it can
FP64_PEAK_TFLOPS = 1.25


def run_shapes_f64(args) -> list:
    """--shapes with --dtype f64, c64 or c128: the double-precision (DPOTRF)
    or the complex Hermitian (CPOTRF, ZPOTRF) factorization of
    A = G G^H / n + I (G iid normal, complex for c64 / c128; 64 distinct
    matrices repeated), the same timing as run_shapes; f64 and c128 against
    the measured FP64 rate, c64 against the FP32 roofline (complex: 4 n^3 / 3
    real flops a matrix)."""
    import torch

    import matrix_dense_linear_gb300 as bl
    import synth
    bl.library()
    dev = torch.device("cuda", 0)
    cplx = args.dtype in ("c64", "c128")
    if args.dtype == "c64":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        peak = sms * 128 * 2 * peaks()["sm_max_mhz"] * 1e6 / 1e12
        peak_src = "FP32: SMs x 128 FMA x 2 x max clock"
    else:
        try:
            peak, peak_src = bl.fma_probe(64), "measured (bl_fma_probe)"
        except Exception:  # noqa: BLE001
            peak, peak_src = FP64_PEAK_TFLOPS, "nominal"
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    rows = []
    for spec in args.shapes.split(","):
        n, batch = (int(x) for x in spec.lower().split("x"))
        distinct = min(batch, 64)
        if cplx:
            mats = []
            for b in range(distinct):
                g = synth.rng(7, b)
                G = g.standard_normal((n, n)) + 1j * g.standard_normal((n, n))
                mats.append((G @ G.conj().T / n + np.eye(n)).astype(
                    np.complex64 if args.dtype == "c64" else np.complex128))
        else:
            mats = [synth.gram(n, synth.rng(6, b), "normal", float(n), 1.0)
                    for b in range(distinct)]
        one = np.concatenate([np.asfortranarray(m).ravel(order="F") for m in mats])
        buf = np.tile(one, -(-batch // distinct))[: batch * n * n]
        src = torch.from_numpy(np.ascontiguousarray(buf)).to(dev)
        nbytes = src.numel() * src.element_size()
        nrep = int(max(1, min(max(args.steps, -(-2 * l2 // nbytes)),
                              REPLICA_CAP_BYTES // max(nbytes, 1))))
        reps = torch.empty((nrep, src.numel()), dtype=src.dtype, device=dev)
        fac = bl.factor_complex if cplx else bl.factor_double
        info = torch.zeros(batch, dtype=torch.int32, device=dev)
        st = torch.cuda.current_stream()
        for i in range(min(args.warmup, nrep)):
            reps[i].copy_(src)
            fac(reps[i], n, n, n * n, batch, info, st, uplo=args.uplo)
        torch.cuda.synchronize()
        k = min(args.steps, nrep)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(k):
                fac(reps[i], n, n, n * n, batch, info, torch.cuda.current_stream(),
                    uplo=args.uplo)
        ts = []
        for _ in range(3):
            for i in range(k):
                reps[i].copy_(src)
            flush.fill_(1.0)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(st)
            g.replay()
            e1.record(st)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / k)
        assert not info.cpu().numpy().any()
        ms = statistics.median(ts)
        tflops = (4 if cplx else 1) * flops_per_matrix(n) * batch / (ms / 1e3) / 1e12
        row = {"shape": spec, "dtype": args.dtype, "uplo": args.uplo, "n": n, "batch": batch,
               "ms_per_call": ms, "us_per_call": ms * 1e3, "matrices_per_s": batch / (ms / 1e3),
               "tflops": tflops,
               "roofline": {"bound": "alu", "peak": peak, "unit": "TFLOP/s",
                            "frac": tflops / peak, "peak_source": peak_src},
               "calls_timed": k}
        print(json.dumps(row), flush=True)
        rows.append(row)
        del reps, g
        torch.cuda.empty_cache()
    return rows


def run_potrs(args) -> dict:
    """Batched SPOTRS (solve with the factor) on a workload's factors: the
    batch is factored once on the device, then each timed step solves nrhs
    right-hand sides per system on its own cold replica of B (L2 flushed
    outside the timed region). Work per system: 2 n^2 nrhs flops; bytes: the
    factor's lower triangle read, B read and X written."""
    import torch

    import matrix_dense_linear_gb300 as bl
    bl.library()
    dev = torch.device("cuda", 0)
    pk = peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    bt = make_host_batch(args.workload, args.batch)
    n, batch, nrhs = bt.n, bt.batch, args.nrhs
    dA = torch.from_numpy(bt.buf).to(dev)
    info = torch.zeros(batch, dtype=torch.int32, device=dev)
    bl.factor(dA, n, bt.lda, bt.strideA, batch, info)
    torch.cuda.synchronize()
    assert not info.cpu().numpy().any()
    g = np.random.default_rng(7)
    span = batch * n * nrhs
    Bh = torch.from_numpy(g.standard_normal(span).astype(np.float32))
    pristine = Bh.to(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nrep = int(max(1, min(max(args.steps, -(-2 * l2 // (4 * span))),
                          REPLICA_CAP_BYTES // (4 * span))))
    reps = torch.empty((nrep, span), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def call(i, st):
        code = bl.spotrs_batched(dA, n, bt.lda, bt.strideA, reps[i], nrhs, n, n * nrhs, batch,
                                 st)
        if code:
            raise bl.BLError(code, "spotrs")

    st = torch.cuda.current_stream()
    for i in range(min(args.warmup, nrep)):
        reps[i].copy_(pristine)
        call(i, st.cuda_stream)
    torch.cuda.synchronize()
    total, done = 0.0, 0
    while done < args.steps:
        chunk = min(nrep, args.steps - done)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            cs = torch.cuda.current_stream().cuda_stream
            for i in range(chunk):
                call(i, cs)
        for i in range(chunk):
            reps[i].copy_(pristine)
        flush.fill_(1.0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        gr.replay()
        e1.record(st)
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
        done += chunk
        del gr
    ms = total / args.steps
    t = ms / 1e3
    flops = 2.0 * n * n * nrhs * batch
    bytes_ = (2.0 * n * (n + 1) + 8.0 * n * nrhs) * batch
    fp32 = sms * 128 * 2 * pk["sm_max_mhz"] * 1e6
    t_hbm, t_alu = bytes_ / (pk["hbm_gbs"] * 1e9), flops / fp32
    if t_hbm >= t_alu:
        roof = {"bound": "hbm", "achieved": bytes_ / t / 1e9, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": bytes_ / t / 1e9 / pk["hbm_gbs"]}
    else:
        roof = {"bound": "alu", "achieved": flops / t / 1e12, "peak": fp32 / 1e12,
                "unit": "TFLOP/s", "frac": flops / t / fp32}
    return {"op": "potrs", "metric": "batched SPOTRS systems/s", "value": batch / t,
            "unit": "systems/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "dtype": "f32", "data": "synthetic",
            "gflops": flops / t / 1e9, "roofline": roof,
            "config": {"workload": f"{args.workload} factors, {nrhs} right-hand sides each",
                       "n": n, "batch": batch, "nrhs": nrhs,
                       "l2": "flushed before each timed chunk; every step solves into its own "
                             "replica of B",
                       "timing": "CUDA events around the replay of a CUDA graph of the K calls"},
            "gpu_launches": args.steps}


def run_reference(args) -> dict:
    """The oracle as it stands, timed on the host cores, on the same workload:
    each step is one pass over a bounded sample of the batch."""
    import oracle
    import synth
    bt = make_host_batch(args.workload, args.batch)
    m = oracle_sample_size(bt.n) or bt.batch
    idx = None if m == bt.batch else list(range(m))
    th = oracle.default_threads()
    for _ in range(args.warmup):
        oracle.potrf_batched(bt.buf, bt.n, bt.lda, bt.strideA, bt.batch, indices=idx, nthreads=th)
    t0 = time.perf_counter()
    used = th
    for _ in range(args.steps):
        _, _, used = oracle.potrf_batched(bt.buf, bt.n, bt.lda, bt.strideA, bt.batch,
                                          indices=idx, nthreads=th)
    dt = time.perf_counter() - t0
    value = args.steps * m / dt
    sample = f"{m} of {bt.batch} matrices (n={bt.n}) per step on {used} host threads"
    w_desc = synth.WORKLOADS[args.workload]
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: n={bt.n}, batch={bt.batch}, lda={bt.lda}, "
                               f"strideA={bt.strideA}, {w_desc.kind} SPD",
                   "n": bt.n, "batch": bt.batch, "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="n64", choices=["n32", "n64", "n128", "n256", "n1024"])
    ap.add_argument("--soak", type=float, default=1.5, help="untimed seconds before timing")
    ap.add_argument("--batch", type=int, default=None,
                    help="factor only the first B matrices of the workload (profiling)")
    ap.add_argument("--no-per-n", dest="per_n", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--op", choices=["potrf", "potrs"], default="potrf",
                    help="potrs: time the solve with the factor instead (one JSON line)")
    ap.add_argument("--nrhs", type=int, default=16, help="right-hand sides per system (potrs)")
    ap.add_argument("--sweep", action="store_true",
                    help="batch sweep of n = 32, 64, 128 (one JSON line per point)")
    ap.add_argument("--shapes", default=None, metavar="NxB,...",
                    help="time these (n, batch) shapes (one JSON line each); 'pages' = "
                         "the shapes the pages quote timings for")
    ap.add_argument("--dtype", choices=["f32", "f64", "c64", "c128"], default="f32",
                    help="f64 / c64 / c128: time the double / complex / double complex "
                         "factorization for --shapes")
    ap.add_argument("--ws", action="store_true",
                    help="--shapes through bl_spotrf_batched_ws (a caller workspace)")
    ap.add_argument("--route", type=int, default=0,
                    help="--shapes: force a route (bl_spotrf_batched_ex): 3 the right-looking "
                         "blocked schedule, 5 the left-looking one; 0 the automatic choice")
    ap.add_argument("--uplo", choices=["L", "U"], default="L",
                    help="storage of the factor for --shapes (U: upper triangle)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.sweep:
        run_sweep(args)
        return
    if args.shapes:
        if args.shapes == "pages":
            args.shapes = PAGES_SHAPES
        if args.dtype in ("f64", "c64", "c128"):
            run_shapes_f64(args)
        else:
            run_shapes(args)
        return
    if args.op == "potrs":
        print(json.dumps(run_potrs(args)), flush=True)
        return

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    barrier = lambda: None  # noqa: E731
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
        barrier = dist.barrier
    out = run_ours(args, rank, world, barrier)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
