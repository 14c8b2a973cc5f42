"""Builds the CUDA library ``libjfa.so`` in-tree with nvcc for sm_103a.

Every translation unit under ``csrc/`` is compiled in parallel into
``_build/`` and linked into ``varlen_flashattention_gb300/libjfa.so``. A unit
is recompiled only when it or a header is newer than its object file.

Two variants of the same sources serve debugging (``build(variant=...)``):
``trace`` (-DJFA_TRACE: per-role event records, libjfa_trace.so) and
``debug`` (-DJFA_DEBUG: bounds checks of every tile load, libjfa_debug.so).
They build into ``_build/<variant>/``; the package loads one of them instead
of libjfa.so when JFA_LIBRARY_VARIANT names it.
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
LIB = os.path.join(PKG, "libjfa.so")
VARIANTS = {"trace": ["-DJFA_TRACE"], "debug": ["-DJFA_DEBUG"]}


def lib_path(variant=None) -> str:
    return LIB if not variant else os.path.join(PKG, f"libjfa_{variant}.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(src: str, obj: str, newest_header: float) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return os.path.getmtime(src) > t or newest_header > t


def build(verbose: bool = False, force: bool = False, extra_flags=None, variant=None) -> str:
    """Compile and link; returns the path of the shared library."""
    if variant is not None and variant not in VARIANTS:
        raise ValueError(f"unknown variant {variant!r} (known: {sorted(VARIANTS)})")
    bdir = BUILD if variant is None else os.path.join(BUILD, variant)
    lib = lib_path(variant)
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest = max([os.path.getmtime(h) for h in _headers()] + [0.0])
    flags = NVCC_FLAGS + VARIANTS.get(variant, []) + list(extra_flags or [])
    jobs = []
    for s in srcs:
        obj = os.path.join(bdir, os.path.basename(s)[:-3] + ".o")
        if force or _stale(s, obj, newest):
            jobs.append((s, obj))

    def compile_one(job):
        s, obj = job
        cmd = [nvcc()] + ARCH + flags + ["-c", s, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(s)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            list(ex.map(compile_one, jobs))
    objs = [os.path.join(bdir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    if jobs or not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        cmd = [nvcc()] + ARCH + ["-shared", "-o", lib] + objs
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib


if __name__ == "__main__":
    v = next((a for a in sys.argv[1:] if a in VARIANTS), None)
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, variant=v))
