"""Builds the CUDA library libulysses.so in this package directory (sm_103a only).

Sources: csrc/*.cu.  Objects go to _build/ beside this file and are reused while they are
newer than their source and every header.  nvcc runs once per translation unit, in
parallel.  No cmake, no torch extension machinery: the library has a plain C ABI.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libulysses.so")
# the debug build (-DULY_DEBUG): kernels bounds-check every global index they compute
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libulysses_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libulysses.so")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(ROOT, "include", "ulysses.h")]


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link; returns the path of libulysses.so (libulysses_debug.so when debug)."""
    BUILD, LIB = (BUILD_DEBUG, LIB_DEBUG) if debug else (globals()["BUILD"], globals()["LIB"])
    flags = NVCC_FLAGS + (["-DULY_DEBUG"] if debug else [])
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest_hdr = max(os.path.getmtime(h) for h in _headers())
    jobs = []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        stale = force or not os.path.exists(obj) or \
            os.path.getmtime(obj) < max(os.path.getmtime(src), newest_hdr)
        jobs.append((src, obj, stale))

    def compile_one(job):
        src, obj, stale = job
        if not stale:
            return src, ""
        tmp = obj + ".tmp%d" % os.getpid()
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", tmp]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, res.stdout, res.stderr))
        os.replace(tmp, obj)
        return src, res.stdout + res.stderr

    with cf.ThreadPoolExecutor(max_workers=len(jobs) or 1) as ex:
        logs = list(ex.map(compile_one, jobs))
    if verbose:
        for src, log in logs:
            if log:
                print("== %s\n%s" % (os.path.basename(src), log))
    objs = [o for _, o, _ in jobs]
    relink = force or not os.path.exists(LIB) or \
        os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs)
    if relink:
        tmp = LIB + ".tmp%d" % os.getpid()
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-ldl"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n%s%s" % (res.stdout, res.stderr))
        os.replace(tmp, LIB)
    return LIB


def build_both(force: bool = False) -> str:
    """The release and the debug library, compiled together (one pool of nvcc processes)."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        rel = ex.submit(build, force)
        dbg = ex.submit(build, force, False, True)
        dbg.result()
        return rel.result()


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
