"""Comparisons shared by the tests: tolerances, reconstruction, untouched memory."""
from __future__ import annotations

import os

import numpy as np

_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_tolerances() -> dict:
    vals = {}
    with open(os.path.join(_GOLDEN, "tolerances.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            vals[k] = float(v)
    return vals


TOL = _read_tolerances()
RECON_PER_N = TOL["recon_budget_per_n"]
MAXREL_PER_N = TOL["max_rel_per_n"]


def sym_from_lower(low: np.ndarray) -> np.ndarray:
    """Full symmetric float64 matrix that a lower triangle defines."""
    low = np.tril(np.asarray(low, dtype=np.float64))
    return low + np.tril(low, -1).T


def recon_error(L: np.ndarray, A_lower: np.ndarray) -> float:
    """||L L^T - A||_F / ||A||_F in float64 over the full symmetric A."""
    L = np.tril(np.asarray(L, dtype=np.float64))
    A = sym_from_lower(A_lower)
    return float(np.linalg.norm(L @ L.T - A) / np.linalg.norm(A))


def max_rel(L: np.ndarray, L_ref: np.ndarray) -> float:
    """max |L - L_ref| / max |L_ref| over the lower triangles, in float64."""
    L = np.tril(np.asarray(L, dtype=np.float64))
    R = np.tril(np.asarray(L_ref, dtype=np.float64))
    den = np.max(np.abs(R))
    return float(np.max(np.abs(L - R)) / den) if den > 0 else float(np.max(np.abs(L - R)))


def check_factor(L_gpu: np.ndarray, L_ref: np.ndarray, info_gpu: int, info_ref: int,
                 A_lower: np.ndarray, what: str = "") -> None:
    """Parity of one matrix: info bit-exact; L within tolerance of the oracle and
    the reconstruction within budget (SPD), or the leading block only (failed)."""
    n = L_ref.shape[0]
    assert int(info_gpu) == int(info_ref), f"{what}: info {info_gpu} != oracle {info_ref}"
    if info_ref == 0:
        if n == 0:
            return
        e = max_rel(L_gpu, L_ref)
        assert e <= MAXREL_PER_N * n, f"{what}: max rel {e:.3e} > {MAXREL_PER_N * n:.3e}"
        r = recon_error(L_gpu, A_lower)
        assert r <= RECON_PER_N * n, f"{what}: recon {r:.3e} > {RECON_PER_N * n:.3e}"
    else:
        k = int(info_ref) - 1  # leading k x k block is defined
        if k > 0:
            e = max_rel(L_gpu[:k, :k], L_ref[:k, :k])
            assert e <= MAXREL_PER_N * max(k, 1), f"{what}: leading block rel {e:.3e}"


def assert_untouched(after: np.ndarray, before: np.ndarray, outside: np.ndarray, what: str = ""):
    """Bitwise equality of every element outside the lower triangles."""
    a = after.view(np.uint32)[outside]
    b = before.view(np.uint32)[outside]
    bad = np.nonzero(a != b)[0]
    assert bad.size == 0, f"{what}: {bad.size} elements outside the lower triangles changed"
