"""In-tree build of libmxfp4.so for sm_103a (nvcc, no cmake).

Each .cu under csrc/ is compiled in parallel to an object under _build/, then
linked into mxfp4_dequant_matmul_gb300/libmxfp4.so.  Rebuilds only what is
older than its sources (any header change rebuilds everything).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmxfp4.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# No --use_fast_math and no -ftz: the E8M0 scale 2^-127 is a subnormal that
# must survive, and every division/expf must be the IEEE/accurate version.
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the MXFP4 CUDA library cannot be built")
    return path


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def headers() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _mtime(p: str) -> float:
    return os.path.getmtime(p) if os.path.exists(p) else -1.0


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    hdr_time = max((_mtime(h) for h in headers()), default=0.0)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    todo, objs = [], []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or verbose_ptxas or _mtime(obj) < max(_mtime(src), hdr_time):
            todo.append((src, obj))

    def compile_one(item):
        src, obj = item
        cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        return r.stderr

    logs = []
    if todo:
        with ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            logs = list(ex.map(compile_one, todo))
    if todo or force or _mtime(LIB) < max(_mtime(o) for o in objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libmxfp4.so failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    if verbose_ptxas:
        for (src, _), log in zip(todo, logs):
            print(f"== {os.path.basename(src)}\n{log}")
    return LIB


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)
