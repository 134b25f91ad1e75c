"""Compile the CUDA sources into the in-tree shared library
``triangular_solve_gb300/_build/libtrsm_gb300.so`` (sm_103a only).

Each translation unit compiles in parallel with nvcc; the objects are then
linked with the static CUDA runtime.  Rebuilds only what changed.

Usage:  python -m triangular_solve_gb300.build [--force] [--verbose-ptxas]
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libtrsm_gb300.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtrsm_gb300.so")


def _deps() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def _compile(src: str, obj: str, extra: list[str]) -> tuple[str, str]:
    tmp = obj + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    os.replace(tmp, obj)  # atomic: concurrent builders never see a partial object
    return src, r.stderr


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest_dep = max([os.path.getmtime(p) for p in _deps()] + [0])
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    todo = []
    objs = []
    for s in srcs:
        o = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or verbose_ptxas or not os.path.exists(o) or \
                os.path.getmtime(o) < max(os.path.getmtime(s), newest_dep):
            todo.append((s, o))
    logs = []
    if todo:
        jobs = jobs or min(len(todo), os.cpu_count() or 4)
        with cf.ThreadPoolExecutor(jobs) as ex:
            for src, err in ex.map(lambda so: _compile(so[0], so[1], extra), todo):
                if err.strip():
                    logs.append(f"== {os.path.basename(src)}\n{err}")
    if todo or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    if verbose_ptxas:
        print("\n".join(logs))
    return LIB


if __name__ == "__main__":
    out = build(force="--force" in sys.argv, verbose_ptxas="--verbose-ptxas" in sys.argv)
    print(out)
