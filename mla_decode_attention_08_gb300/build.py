"""Builds libmla_decode.so in-tree with nvcc for sm_103a (no CMake, no torch).

Each translation unit compiles in parallel into ``_build/``; the shared
library lands next to this file, where the binding loads it.  ``debug=True``
builds ``libmla_decode_debug.so`` (objects in ``_build_debug/``) with
``-DMLA_DEBUG``: the kernels then check their global stores, query loads, tile
coordinates and combine indices against their buffers and report a failed
check as MLA_DERR_DEBUG_BOUNDS instead of making the access.
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
LIB = os.path.join(PKG, "libmla_decode.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libmla_decode_debug.so")
BUILD_TRACE = os.path.join(PKG, "_build_trace")
LIB_TRACE = os.path.join(PKG, "libmla_decode_trace.so")
SOURCES = ["stage1.cu", "stage2.cu", "fp8_quant.cu", "mxfp4_quant.cu", "api.cu", "static_scratch.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmla_decode")
    return exe


def _flags():
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", os.path.join(ROOT, "include")]


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, debug: bool = False,
          trace: bool = False) -> str:
    """Compile (if anything changed) and return the path of the shared library.

    ``trace=True`` builds ``libmla_decode_trace.so`` with ``-DMLA_TRACE``: the
    kernels stamp their start-up milestones (``mla_decode_trace_read``)."""
    if debug and trace:
        raise ValueError("build either the debug or the trace variant")
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else ((BUILD_TRACE, LIB_TRACE) if trace
                                                             else (BUILD, LIB))
    extra = ["-DMLA_DEBUG"] if debug else (["-DMLA_TRACE"] if trace else [])
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(ROOT, "include", "mla_decode.h"))
    exe = nvcc()

    def compile_one(src: str) -> str:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        if force or _stale(o, [s] + headers):
            cmd = [exe] + _flags() + extra + ["-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd), flush=True)
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return o

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(lib, objs):
        cmd = [exe] + ARCH + ["-shared", "-o", lib] + objs + ["-cudart", "static"]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv, debug="--debug" in sys.argv,
                trace="--trace" in sys.argv))
