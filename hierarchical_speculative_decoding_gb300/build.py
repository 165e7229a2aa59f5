"""In-tree build of libtriforce_attn.so for sm_103a (nvcc, no cmake).

Each .cu under csrc/ compiles to an object in parallel, then one shared
library is linked next to this file.  Rebuilds only when a source or header
is newer than the library.  Processes that build at the same time (one per
rank under torchrun) take turns on a file lock; whoever waited finds the
library fresh and returns it without compiling again.

build(debug=True) makes the checked variant, libtriforce_attn_debug.so,
compiled with -DTF_DEBUG: every data-dependent gather index is checked
against its buffer before the access, and violations are collected in device
words that tf_debug_status() reports.
"""

from __future__ import annotations

import concurrent.futures as cf
import fcntl
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtriforce_attn.so")
LIB_DEBUG = os.path.join(PKG, "libtriforce_attn_debug.so")
LOCK = os.path.join(BUILD, ".build.lock")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtriforce_attn.so")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def library(debug: bool = False) -> str:
    return LIB_DEBUG if debug else LIB


def up_to_date(debug: bool = False) -> bool:
    lib = library(debug)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None, debug: bool = False) -> str:
    if not force and up_to_date(debug):
        return library(debug)
    os.makedirs(BUILD, exist_ok=True)
    with open(LOCK, "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)  # one build at a time, across processes
        try:
            if not force and up_to_date(debug):  # built by another process while this one waited
                return library(debug)
            return _compile_and_link(verbose, extra, debug)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _compile_and_link(verbose: bool, extra: list[str] | None, debug: bool = False) -> str:
    cc = nvcc()
    extra = list(extra or []) + (["-DTF_DEBUG"] if debug else [])
    objdir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(objdir, exist_ok=True)
    LIB = library(debug)

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = f"{LIB}.{os.getpid()}.tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        if os.path.exists(tmp):
            os.remove(tmp)
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra=["-Xptxas", "-v"] if "--ptxas" in sys.argv else None, debug="--debug" in sys.argv))
