"""Build the sm_103a CUDA library in-tree: precision_matmul_gb300/_build/libfp8mm.so.

nvcc compiles the kernel instantiations and the C-ABI host code for
``arch=compute_103a,code=sm_103a`` only, with line info for profiling.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libfp8mm.so")
SOURCES = ["fp8mm_host.cu", "fp8mm_aux.cu", "fp8mm_inst_narrow.cu", "fp8mm_inst_fast128.cu", "fp8mm_inst_fast256.cu",
           "fp8mm_inst_pair.cu", "fp8mm_inst_slow.cu", "fp8mm_inst_slow_wide.cu", "fp8mm_inst_slow_pair.cu", "fp8mm_inst_slow_held.cu", "fp8mm_inst_mx.cu", "fp8mm_inst_mx_wide.cu",
           "fp8mm_inst_f4.cu"]
HEADERS = ["fp8mm_kernel.cuh", "fp8mm_kernels.h", "ptx.cuh"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    cand = [os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "fp8mm.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit in parallel, then link the shared library."""
    if not force and not _stale():
        return LIB
    from concurrent.futures import ThreadPoolExecutor
    os.makedirs(BUILD, exist_ok=True)
    nvcc = nvcc_path()
    common = ["-std=c++17", "-O3", ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
              "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]
    if verbose:
        common.insert(0, "-Xptxas=-v")

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + f".{os.getpid()}.o")
        subprocess.run([nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj], check=True)
        return obj

    workers = max(1, min(len(SOURCES), os.cpu_count() or 1))
    objs = [os.path.join(BUILD, os.path.splitext(src)[0] + f".{os.getpid()}.o") for src in SOURCES]
    try:
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(compile_one, SOURCES))
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run([nvcc, ARCH, "-shared", *objs, "-o", tmp], check=True)
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
