"""Build the KDA CUDA library (libkda.so) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libkda.so")
SOURCES = [os.path.join(CSRC, "kda_fwd.cu")]
HEADERS = [os.path.join(CSRC, h) for h in ("ptx.cuh", "kda_common.cuh", "kda_chunk.cuh", "kda_fwd_mma.cuh", "kda_fwd_mma32.cuh", "tcgen05.cuh", "kda_fwd_tc.cuh", "kda_probe.cuh", "kda_decode.cuh")] + [os.path.join(INCLUDE, "kda.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def command(out: str = LIB, extra=()) -> list:
    return [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
            "-shared", "-I", INCLUDE, *extra, "-o", out, *SOURCES]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in SOURCES + HEADERS)


def build_library(force: bool = False, verbose: bool = False) -> str:
    if force or stale():
        tmp = LIB + ".%d.tmp" % os.getpid()
        extra = ["-Xptxas", "-v"] if verbose else []
        subprocess.run(command(tmp, extra), check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
