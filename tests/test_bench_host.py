"""Host-side arithmetic of bench.py (no GPU): the roofline's byte counts, the
launch count it claims per call against the library's own route rule, and the
traffic figures' source check."""
from __future__ import annotations

import math

import pytest

import bench


def _sectors_brute(n: int) -> int:
    """Bytes the lower triangle moves in 32-byte sectors, in and out, for
    columns starting on a sector: enumerate every element's sector."""
    touched = 0
    for k in range(n):
        sectors = {(4 * i) // 32 for i in range(k, n)}
        touched += len(sectors)
    return 2 * 32 * touched


@pytest.mark.parametrize("n", [1, 2, 7, 8, 9, 31, 32, 33, 64, 100, 128])
def test_sector_bytes_match_a_brute_force_count(n):
    assert bench.sector_bytes_per_matrix(n) == _sectors_brute(n)


def test_sector_bytes_at_n32_and_algorithmic_bytes():
    # the n = 32 figure the workload table quotes: 5120 bytes, against 4224
    # algorithmic (the lower triangle in and out, 4 n (n + 1))
    assert bench.sector_bytes_per_matrix(32) == 5120
    for n in (1, 32, 64, 1024):
        assert bench.alg_bytes_per_matrix(n) == 4 * n * (n + 1)
        assert bench.flops_per_matrix(n) == n ** 3 / 3


@pytest.mark.parametrize("n,batch", [(32, 1024), (128, 1024), (129, 8), (256, 4096),
                                     (384, 512), (1024, 1), (1024, 128), (1024, 512),
                                     (2048, 64), (2048, 128), (4096, 8)])
def test_launch_count_follows_the_library_route(n, batch):
    import matrix_dense_linear_gb300 as bl
    panels = math.ceil(n / 128)
    got = bench.launches_per_call(n, batch)
    route = bl.route(n, batch)
    if n <= 128:
        assert route in (bl.ROUTE_WARP, bl.ROUTE_CTA) and got == 1
    elif route == bl.ROUTE_LEFT:
        # per panel: its update (not the first), its factor, its solve (not the last)
        assert got == 3 * panels - 2
    else:
        assert route == bl.ROUTE_BLOCKED
        # right-looking: a factor per panel, a solve per panel but the last,
        # and an update for each of those unless fused into the solve
        assert panels + (panels - 1) <= got <= panels + 2 * (panels - 1)


def test_roofline_bound_and_fraction():
    pk = {"hbm_gbs": 6684.5, "sm_max_mhz": 2070.0}
    r = bench.roofline_entry("n32", 32, 1024, 0.005, pk, 152)
    assert r["bound"] == "hbm"
    assert r["frac"] == pytest.approx(4224 * 1024 / 5e-6 / 1e9 / 6684.5)
    assert r["frac_sector_rounded"] == pytest.approx(r["frac"] * 5120 / 4224)
    r = bench.roofline_entry("n1024", 1024, 512, 2.4, pk, 152)
    assert r["bound"] == "alu" and "frac_sector_rounded" not in r
    peak = 152 * 128 * 2 * 2070e6 / 1e12
    assert r["frac"] == pytest.approx(1024 ** 3 / 3 * 512 / 2.4e-3 / 1e12 / peak)


def test_traffic_is_null_once_its_sources_change(monkeypatch):
    srcs, sha, nbytes, scope = bench.TRAFFIC["n64"]
    assert bench.traffic_for("n64", 64) == nbytes  # the committed sources
    monkeypatch.setitem(bench.TRAFFIC, "n64", (srcs, "0" * 16, nbytes, scope))
    assert bench.traffic_for("n64", 64) is None
    assert bench.traffic_for("no-such-workload", 64) is None


def test_traffic_is_null_off_the_captured_batch():
    # the figures were captured on each workload's own batch; another batch
    # (bench.py --batch) does not rescale them
    for name, (_, _, nbytes, _) in bench.TRAFFIC.items():
        n = int(name[1:])
        batch = {"n32": 1024, "n64": 1024, "n128": 1024, "n256": 4096, "n1024": 512}[name]
        assert bench.traffic_for(name, n, batch) == nbytes
        assert bench.traffic_for(name, n, batch // 2) is None
        assert bench.traffic_for(name, n + 1, batch) is None
