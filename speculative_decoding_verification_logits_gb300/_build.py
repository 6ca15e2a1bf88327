"""Compiles the CUDA library (csrc/*.cu) into libsdverify.so, in-tree, for
sm_103a only.  Used by ``__graft_entry__.build()`` and on first import."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libsdverify.so")
SOURCES = sorted(glob.glob(os.path.join(PKG, "csrc", "*.cu")))
HEADERS = sorted(glob.glob(os.path.join(PKG, "csrc", "*.cuh")) +
                 glob.glob(os.path.join(ROOT, "include", "*.h")))

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Each translation unit is compiled to an object in parallel, then the
    objects are linked into the shared library."""
    if not force and not stale():
        return LIB
    tag = f".tmp{os.getpid()}"
    nvc = nvcc()
    base = [nvc, *NVCC_FLAGS, "-I", os.path.join(ROOT, "include")]
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.join(PKG, os.path.basename(src) + tag + ".o")
        cmd = [*base, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        objs.append(obj)
        procs.append(subprocess.Popen(cmd))
    try:
        rcs = [p.wait() for p in procs]
        if any(rcs):
            raise subprocess.CalledProcessError(next(r for r in rcs if r), "nvcc -c")
        tmp = LIB + tag
        # -ldl: the NVTX ranges look up a profiler's injection library by dlopen
        link = [nvc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", *objs, "-ldl",
                "-o", tmp]
        if verbose:
            print(" ".join(link), flush=True)
        subprocess.run(link, check=True)
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB
