"""In-tree build of the C-ABI library ``libspmv_gb300.so`` for sm_103a.

The translation units (host planner and converters, CSR tile kernel, CSR
segment kernel, DELTA kernel, sliced-ELL kernel, matrix-free FEM kernel,
conjugate-gradient kernels, allocation-free entry point) are compiled in parallel with nvcc
and linked into one shared object next to this file.
Usage: ``python -m sparse_matrix_vector_gb300.build`` or ``build_library()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libspmv_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["spmv_host.cpp", "spmv_csr.cu", "spmv_csr_seg.cu", "spmv_delta.cu", "spmv_sell.cu",
           "spmv_fem.cu", "spmv_pcg.cu", "spmv_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "--expt-relaxed-constexpr"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    return os.path.join(cuda, "bin", "nvcc")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(INCLUDE, "spmv.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def up_to_date() -> bool:
    return (os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= _newest_input())


# The checked build (SPMV_CHECKED=1: kernels test indices before use; see
# include/spmv.h, spmv_checked_build), a separate library for debugging.
CHECKED_LIB_PATH = os.path.join(HERE, "libspmv_gb300_checked.so")
CHECKED_BUILD_DIR = os.path.join(HERE, "_build_checked")


def build_library(force: bool = False, verbose: bool = False,
                  extra_flags: list[str] | None = None, checked: bool = False) -> str:
    """Compile and link the library (or its checked build) if any input is
    newer. Returns its path."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    build_dir = CHECKED_BUILD_DIR if checked else BUILD_DIR
    if (not force and not extra_flags and os.path.exists(lib_path)
            and os.path.getmtime(lib_path) >= _newest_input()):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = nvcc_path()
    flags = (NVCC_FLAGS + ARCH + ["-I", INCLUDE] + (["-DSPMV_CHECKED=1"] if checked else [])
             + list(extra_flags or []))

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        objs = list(pool.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))
