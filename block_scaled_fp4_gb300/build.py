"""Builds the in-tree CUDA library ``_build/libqmoe.so`` for sm_103a with nvcc.

Each ``csrc/*.cu`` is compiled in parallel, then linked into one shared
library (CUDA runtime linked statically).  ``build()`` recompiles only what is
older than its sources or headers."""
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
LIB = os.path.join(BUILD, "libqmoe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", f"-I{os.path.join(ROOT, 'include')}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the QMoE CUDA library cannot be built")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in sources]

    def compile_one(src_obj):
        src, obj = src_obj
        if not _stale(obj, [src] + headers):
            return obj, ""
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, len(sources))) as ex:
        for obj, log in ex.map(compile_one, zip(sources, objs)):
            if verbose and log:
                print(log)
    if _stale(LIB, objs):
        cmd = [nvcc, *ARCH, "-shared", "-o", LIB + ".tmp", *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
