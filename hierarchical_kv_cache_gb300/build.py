"""Builds the in-tree C-ABI library ``libhicache_gb300.so`` for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel (CUDA sources
with nvcc for ``compute_103a``/``sm_103a`` only, plain C++ with g++), then
linked into one shared library next to this file.  Nothing is installed into
site-packages; the binding loads the library from this directory.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import time

HERE = os.path.dirname(os.path.abspath(__file__))
REPO = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(REPO, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libhicache_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def _compile_cmd(src: str, obj: str, ptxas_verbose: bool):
    cuda = _cuda_home()
    inc = ["-I", INCLUDE, "-I", CSRC, "-I", os.path.join(cuda, "include")]
    if src.endswith(".cu"):
        cmd = [os.path.join(cuda, "bin", "nvcc"), "-c", src, "-o", obj, "-std=c++17", "-O3",
               "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-Wall", *inc]
        if ptxas_verbose:
            cmd += ["-Xptxas", "-v"]
        return cmd
    return ["g++", "-c", src, "-o", obj, "-std=c++17", "-O3", "-fPIC", "-Wall", "-Wextra", *inc]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _sources() + _headers() + [__file__])


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    """Compile and link the library; returns its path.

    Processes that build at the same time (the ranks of a multi-GPU run, parallel
    test workers) take turns on a lock file, and a process that finds the library
    current once it holds the lock does not rebuild it.
    """
    import fcntl

    if not force and not ptxas_verbose and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    asked = time.time()
    with open(os.path.join(BUILD_DIR, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)  # released when the file closes
        # another process may have built it while this one waited
        if (not ptxas_verbose and up_to_date()
                and (not force or os.path.getmtime(LIB_PATH) >= asked)):
            return LIB_PATH
        return _build_locked(ptxas_verbose, quiet)


def _build_locked(ptxas_verbose: bool, quiet: bool) -> str:
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        jobs.append((src, obj, _compile_cmd(src, obj, ptxas_verbose)))

    def run(job):
        src, obj, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compiling {os.path.basename(src)} failed:\n{' '.join(cmd)}\n"
                               f"{r.stdout}\n{r.stderr}")
        return (src, r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(run, jobs))
    if not quiet or ptxas_verbose:
        for src, out in outs:
            if out.strip():
                print(f"--- {os.path.basename(src)}\n{out}")
    cuda = _cuda_home()
    tmp = LIB_PATH + ".tmp"
    link = [os.path.join(cuda, "bin", "nvcc"), "-shared", "-o", tmp, *[j[1] for j in jobs],
            *ARCH, "-cudart", "shared", "-Xlinker", "-rpath," + os.path.join(cuda, "lib64")]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"linking failed:\n{' '.join(link)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys

    print(build(force=True, ptxas_verbose="-v" in sys.argv, quiet=False))
