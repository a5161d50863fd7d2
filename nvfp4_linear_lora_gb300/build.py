"""Builds ``libh3lin.so`` in-tree from ``csrc/*.cu`` for sm_103a (GB300).

    python -m nvfp4_linear_lora_gb300.build        # or build() from Python

Each translation unit is compiled in parallel with nvcc, then linked into one
shared library (CUDA runtime linked statically, no libcuda link: the TMA
encoder is fetched through the runtime's driver entry point).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libh3lin.so")
# The bounds build: the same sources with -DH3LIN_BOUNDS, whose kernels check
# every plain global index and report a bad one in the status word instead of
# touching memory (see h3lin_selftest_bounds in include/h3lin.h).
BOUNDS_LIB = os.path.join(PKG, "libh3lin_bounds.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libh3lin.so")
    return nvcc


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs + [os.path.join(ROOT, "include", "h3lin.h")]


def _compile(src, build_dir, extra, verbose_ptxas=False):
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [_nvcc()] + ARCH + FLAGS + extra + (["-Xptxas", "-v"] if verbose_ptxas else []) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def needs_build(lib=LIB):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _sources() + _headers())


def build(force=False, verbose_ptxas=False, bounds=False):
    """Compile every CUDA source for sm_103a and link ``libh3lin.so`` (with
    ``bounds``: ``libh3lin_bounds.so``, the bounds-checked build)."""
    lib = BOUNDS_LIB if bounds else LIB
    if not force and not needs_build(lib):
        return lib
    build_dir = os.path.join(BUILD, "bounds") if bounds else BUILD
    extra = ["-DH3LIN_BOUNDS"] if bounds else []
    os.makedirs(build_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        results = list(ex.map(lambda s: _compile(s, build_dir, extra, verbose_ptxas), _sources()))
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = lib + ".tmp"
    cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, bounds="--bounds" in sys.argv))
