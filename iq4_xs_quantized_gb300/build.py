"""Build libiq4xs.so in-tree for sm_103a with nvcc (no cmake).

Each translation unit under ``csrc/`` is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3`` and linked into
``iq4_xs_quantized_gb300/libiq4xs.so`` against the shared CUDA runtime.  The
library is rebuilt only when a source or header is newer than it.

``build(bounds_check=True)`` compiles the same sources with
``-DIQ4XS_BOUNDS_CHECK`` into ``libiq4xs_bounds.so`` (objects under
``_build_bounds/``): the debug build whose kernels check every global access,
TMA box origin and computed shared-memory range against its buffer and record
misses in the device error word.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libiq4xs.so")
BOUNDS_LIB = os.path.join(PKG, "libiq4xs_bounds.so")
BOUNDS_BUILD = os.path.join(PKG, "_build_bounds")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xptxas", "-warn-spills"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return cand


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [
        os.path.join(ROOT, "include", "iq4xs.h"), os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, extra, build_dir: str) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc_path(), *ARCH, *NVCC_FLAGS, *extra, "-I", os.path.join(ROOT, "include"),
           "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, bounds_check: bool = False) -> str:
    """Compile and link the library (the bounds-checked one with
    ``bounds_check``); return its path."""
    lib, build_dir = (BOUNDS_LIB, BOUNDS_BUILD) if bounds_check else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if bounds_check:
        extra += ["-DIQ4XS_BOUNDS_CHECK"]
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc_path(), *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                bounds_check="--bounds" in sys.argv))
