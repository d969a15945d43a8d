"""Compile the CUDA sources of this package into ``libmla_gb300.so`` (in-tree).

Each ``csrc/*.cu`` is compiled for sm_103a in its own nvcc process (in
parallel), then the objects are linked into one shared library that shares
the process's CUDA runtime (``-cudart shared``) with PyTorch.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libmla_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
BUILD_DIR = os.path.join(PKG, "_build")
# The checked build (-DMLA_CHECK: index checks in the decode kernels that skip
# an out-of-range access and raise MLA_DEV_BOUNDS), kept beside the default one.
CHECK_LIB_PATH = os.path.join(PKG, "libmla_gb300_check.so")
CHECK_BUILD_DIR = os.path.join(PKG, "_build_check")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-cudart", "shared",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, extra_flags=None, check: bool = False) -> str:
    """Build (if stale) and return the path of the shared library; with
    ``check`` the checked build (compiled with -DMLA_CHECK) instead."""
    build_dir = CHECK_BUILD_DIR if check else BUILD_DIR
    lib_path = CHECK_LIB_PATH if check else LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    flags = ARCH + NVCC_FLAGS + ["-I", INCLUDE, "-I", CSRC] + list(extra_flags or [])
    if check:
        flags.append("-DMLA_CHECK")
    objs = []
    jobs = []
    for s in srcs:
        o = os.path.join(build_dir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append([nvcc(), *flags, "-c", s, "-o", o])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(run, jobs))
    if force or jobs or _stale(lib_path, objs):
        run([nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", lib_path, *objs])
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(verbose=True, force="--force" in sys.argv))
