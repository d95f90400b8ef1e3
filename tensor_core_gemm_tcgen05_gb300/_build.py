"""Build step of the CUDA library: compiles ``csrc/gemm_api.cu`` (with the kernel header)
into ``libgb300gemm.so`` inside the package, for sm_103a only."""
from __future__ import annotations

import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libgb300gemm.so")
SOURCES = [os.path.join(PKG, "csrc", "gemm_api.cu"), os.path.join(PKG, "csrc", "gemm_noalloc.cu")]
DEPS = SOURCES + glob.glob(os.path.join(PKG, "csrc", "*.cuh")) + [os.path.join(ROOT, "include", "gemm.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if it is missing or older than its sources; return its path."""
    stale = force or not os.path.exists(LIB) or any(
        os.path.getmtime(d) > os.path.getmtime(LIB) for d in DEPS)
    if stale:
        tmp = f"{LIB}.tmp{os.getpid()}"
        cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-o", tmp, *SOURCES]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
