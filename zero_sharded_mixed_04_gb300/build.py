"""Builds libzero_gb300.so in the package directory with nvcc for sm_103a,
and libzero_gb300_debug.so: the same sources with -DZERO_DEBUG, whose kernels
check every index range against the buffers' lengths before touching it.

The translation units are compiled in parallel.  The library links the CUDA
runtime statically, so it only needs the driver at run time.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libzero_gb300.so")
DEBUG_BUILD_DIR = os.path.join(BUILD_DIR, "debug")
DEBUG_LIB_PATH = os.path.join(PKG, "libzero_gb300_debug.so")

SOURCES = ["zero_step.cu", "zero3_gather.cu", "zero_host.cpp"]
HEADERS = [os.path.join(INCLUDE, "zero_gb300.h"), os.path.join(CSRC, "zero_common.cuh"),
           os.path.join(CSRC, "zero_elem.cuh"), os.path.join(CSRC, "zero_kernels.cuh")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              f"-I{INCLUDE}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libzero_gb300.so")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    out_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    path = os.path.join(CSRC, src)
    if _stale(obj, [path, *HEADERS]):
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *(["-DZERO_DEBUG"] if debug else []), "-c", path,
               "-o", obj + ".tmp"]
        if verbose and src.endswith(".cu"):
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        os.replace(obj + ".tmp", obj)
    return obj


def _link(target: str, objs: list[str], force: bool) -> None:
    if force or _stale(target, objs):
        tmp = target + f".tmp{os.getpid()}"
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, target)


def build_library(force: bool = False, verbose: bool = False, debug: bool = True) -> str:
    """Compile (if stale) and link libzero_gb300.so, and with ``debug`` also
    libzero_gb300_debug.so (the same sources with -DZERO_DEBUG: device-side
    bounds checks); the translation units compile in parallel.  Returns the
    release library's path."""
    dirs = [BUILD_DIR] + ([DEBUG_BUILD_DIR] if debug else [])
    for d in dirs:
        os.makedirs(d, exist_ok=True)
        if force:
            for f in os.listdir(d):
                p = os.path.join(d, f)
                if os.path.isfile(p):
                    os.remove(p)
    jobs = [(src, False) for src in SOURCES] + ([(src, True) for src in SOURCES] if debug else [])
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(j[0], verbose, j[1]), jobs))
    _link(LIB_PATH, objs[:len(SOURCES)], force)
    if debug:
        _link(DEBUG_LIB_PATH, objs[len(SOURCES):], force)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
