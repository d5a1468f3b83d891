"""Build the CUDA library (``_build/libmoe_int4.so``) with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library exporting the C ABI of ``include/moe_int4.h``.  No CMake; nvcc only.

``build(debug_bounds=True)`` builds a second copy with ``-DMOE_DEBUG_BOUNDS``
(``_build/debug_bounds/libmoe_int4.so``): the kernels check the indices they read
back from routing buffers and record MOE_DEVERR_BOUNDS instead of going out of
range.  ``ops.load_library`` loads it when MOE_INT4_DEBUG_BOUNDS=1.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmoe_int4.so")
DEBUG_BUILD = os.path.join(BUILD, "debug_bounds")
DEBUG_LIB = os.path.join(DEBUG_BUILD, "libmoe_int4.so")
SOURCES = ["abi.cu", "align.cu", "pack.cu", "gemm.cu", "noalloc.cu", "ep.cu", "gemv.cu"]
HEADERS = ["common.cuh", "kernels.cuh", "dequant.cuh", "gemv.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "moe_int4.h"))
    return files


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=None,
          debug_bounds: bool = False) -> str:
    """Compile (if needed) and return the path of the shared library (the
    debug-bounds copy with debug_bounds=True)."""
    out_dir, lib = (DEBUG_BUILD, DEBUG_LIB) if debug_bounds else (BUILD, LIB)
    if not force and not _stale(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + list(extra_flags or []) + (["-DMOE_DEBUG_BOUNDS"] if debug_bounds else [])

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + ARCH + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> None:
    """The library and its debug-bounds copy, compiled side by side."""
    with ThreadPoolExecutor(2) as ex:
        list(ex.map(lambda d: build(force=force, debug_bounds=d), (False, True)))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
