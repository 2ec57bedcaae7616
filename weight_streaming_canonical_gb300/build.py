"""Builds libafx.so in-tree (weight_streaming_canonical_gb300/_build/).

Every translation unit is compiled in parallel, CUDA sources for sm_103a
only, then linked into one shared library with the CUDA runtime linked
statically.  Run as ``python -m weight_streaming_canonical_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libafx.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libafx_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3,-pthread", "--expt-relaxed-constexpr"]
CXX_FLAGS = ["-O3", "-std=c++17", "-fPIC", "-pthread", "-Wall", "-Wextra"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the afx library needs the CUDA toolkit to build")


def _cuda_include(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, debug_bounds: bool = False) -> str:
    """Builds libafx.so; debug_bounds builds libafx_debug.so instead, with
    every buffer bound checked in the kernels (AFX_DEBUG_BOUNDS=1)."""
    build_dir = BUILD_DEBUG if debug_bounds else BUILD
    lib = LIB_DEBUG if debug_bounds else LIB
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(os.path.dirname(HERE), "include", "afx.h"))
    srcs = sources()
    objs = []
    jobs = []
    for src in srcs:
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            defs = ["-DAFX_DEBUG_BOUNDS=1"] if debug_bounds else []
            if src.endswith(".cu"):
                cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defs, "-c", src, "-o", obj]
                if ptxas_info:
                    cmd.insert(1, "-Xptxas=-v")
            else:
                cmd = ["g++", *CXX_FLAGS, *defs, "-I", _cuda_include(nvcc), "-c", src, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0 or (verbose and r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}")

    with cf.ThreadPoolExecutor(max(1, len(jobs))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-pthread", "-lcublas"])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    path = build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv,
                 debug_bounds="--debug-bounds" in sys.argv)
    print(path)
