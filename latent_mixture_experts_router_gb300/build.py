"""Compile the CUDA library in-tree: csrc/*.cu -> liblatent_moe.so (sm_103a only).

Each translation unit compiles in its own nvcc process, in parallel; objects go
to ``_build/`` next to this file.  A unit is recompiled when it or any header
under csrc/ or include/ is newer than its object.

``build(checked=True)`` makes the checked variant liblatent_moe_checked.so (objects
in ``_build_checked/``): the same sources with -DLMOE_BOUNDS_CHECKS=1, whose forward
validates the routing structures before any kernel indexes with them.  It is off by
default; the tests that exercise it build it on demand.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "liblatent_moe.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "liblatent_moe_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _cuda_lib_dirs():
    dirs = []
    for d in ("/usr/local/cuda/lib64", "/usr/local/cuda/lib64/stubs",
              "/usr/local/cuda/targets/sbsa-linux/lib", "/usr/local/cuda/targets/sbsa-linux/lib/stubs",
              "/usr/local/cuda/targets/x86_64-linux/lib", "/usr/local/cuda/targets/x86_64-linux/lib/stubs"):
        if os.path.isdir(d):
            dirs.append("-L" + d)
    return dirs


def _newer(src: str, obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return os.path.getmtime(src) > t or any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Build (or reuse) the shared library and return its path (checked: the bounds-checked
    variant)."""
    BUILD = BUILD_CHECKED if checked else globals()["BUILD"]
    LIB = LIB_CHECKED if checked else globals()["LIB"]
    if checked:
        extra_flags = tuple(extra_flags) + ("-DLMOE_BOUNDS_CHECKS=1",)
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))
    nvcc = _nvcc()
    jobs = []
    for s in srcs:
        obj = os.path.join(BUILD, os.path.basename(s) + ".o")
        if _newer(s, obj, deps):
            jobs.append([nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", s, "-o", obj])
    objs = [os.path.join(BUILD, os.path.basename(s) + ".o") for s in srcs]

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {cmd[-3]}")
    if jobs or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        cmd = [nvcc, *ARCH, "-shared", "-o", LIB, *objs, *_cuda_lib_dirs(), "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("link failed")
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
