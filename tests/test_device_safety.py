"""Safety rules of the CUDA sources, checked on their text (CPU): no kernel
traps or asserts, every wait on an mbarrier is the bounded helper with the
library's cycle budget, and every file that allocates tensor memory also
frees it.
"""
from __future__ import annotations

import glob
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "matrix_dense_linear_gb300", "csrc")
SOURCES = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")))
HELPER = "tc_sm100.cuh"  # the one place the raw wait instructions may appear


def _code(path: str) -> str:
    """The file without its comments."""
    s = open(path).read()
    s = re.sub(r"/\*.*?\*/", "", s, flags=re.S)
    return re.sub(r"//[^\n]*", "", s)


def test_sources_found():
    names = {os.path.basename(p) for p in SOURCES}
    assert HELPER in names and "potrf_warp.cu" in names and len(names) >= 10


def test_no_trap_or_device_assert():
    for p in SOURCES:
        code = _code(p)
        assert "__trap" not in code, p
        assert not re.search(r"\btrap\s*;", code), p
        assert not re.search(r"\bassert\s*\(", code), p


def test_raw_mbarrier_waits_only_in_the_helper():
    for p in SOURCES:
        if os.path.basename(p) == HELPER:
            continue
        code = _code(p)
        assert "mbarrier.try_wait" not in code and "mbarrier.test_wait" not in code, p


def test_every_mbarrier_wait_is_bounded():
    calls = 0
    for p in SOURCES:
        for m in re.finditer(r"mbar_wait\(([^;]*)\)", _code(p)):
            if os.path.basename(p) == HELPER and "max_cycles" in m.group(1):
                continue  # the definition
            calls += 1
            assert "kWaitCycles" in m.group(1), (p, m.group(0))
    assert calls >= 10
    helper = _code(os.path.join(CSRC, HELPER))
    body = helper[helper.index("bool mbar_wait("):]
    body = body[: body.index("\n}\n")]
    assert "clock64() - t0 > max_cycles" in body and "return false" in body


def test_tensor_memory_is_freed_where_allocated():
    files = 0
    for p in SOURCES:
        code = _code(p)
        if os.path.basename(p) == HELPER:
            continue
        assert "tcgen05.alloc" not in code and "tcgen05.dealloc" not in code, p
        allocs = re.findall(r"tmem_alloc\([^,]*,\s*([^)]*)\)", code)
        if not allocs:
            continue
        files += 1
        frees = re.findall(r"tmem_dealloc\([^,]*,\s*([^)]*)\)", code)
        # the same number of columns is released as was allocated
        assert frees and set(frees) == set(allocs), (p, allocs, frees)
    assert files >= 3
