"""Build libbl_spotrf.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` is compiled in parallel to an object under ``_build/``
(``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3 -Xptxas -v``), the
ptxas resource report of every file is kept in ``_build/<file>.ptxas.txt``,
and the objects are linked into ``matrix_dense_linear_gb300/libbl_spotrf.so``.

Usage: ``python -m matrix_dense_linear_gb300.build [--force]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
SO = os.path.join(PKG, "libbl_spotrf.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(SO):
        return False
    t = os.path.getmtime(SO)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str) -> str:
    base = os.path.splitext(os.path.basename(src))[0]
    obj = os.path.join(BUILD, base + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", src, "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(BUILD, base + ".ptxas.txt"), "w") as f:
        f.write(p.stderr)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{p.stdout}\n{p.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if any source changed. Returns the .so path."""
    if not force and up_to_date():
        return SO
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(_compile, srcs))
    tmp = SO + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, SO)
    if verbose:
        print(f"built {SO}")
    return SO


def ptxas_report() -> str:
    """Concatenated ptxas resource reports of the last build (current sources
    only: reports left by a deleted source are ignored)."""
    out = []
    for src in sources():
        f = os.path.join(BUILD, os.path.splitext(os.path.basename(src))[0] + ".ptxas.txt")
        if os.path.exists(f):
            with open(f) as fh:
                out.append(fh.read())
    return "\n".join(out)


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
