"""Build the KDA CUDA library (libkda.so) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libkda.so")
DEBUG_LIB = os.path.join(PKG, "libkda_debug.so")  # the same sources with KDA_DEBUG bounds checks
SOURCES = [os.path.join(CSRC, "kda_fwd.cu")]
HEADERS = [os.path.join(CSRC, h) for h in ("kda_debug.cuh", "ptx.cuh", "kda_common.cuh", "kda_chunk.cuh", "kda_fwd_mma.cuh", "kda_fwd_mma32.cuh", "cluster.cuh", "kda_fwd_shared.cuh", "tcgen05.cuh", "kda_fwd_tc.cuh", "kda_probe.cuh", "kda_decode.cuh")] + [os.path.join(INCLUDE, "kda.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def command(out: str = LIB, extra=()) -> list:
    return [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
            "-shared", "-I", INCLUDE, *extra, "-o", out, *SOURCES]


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in SOURCES + HEADERS)


def build_library(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    if force or stale(lib):
        tmp = lib + ".%d.tmp" % os.getpid()
        extra = (["-Xptxas", "-v"] if verbose else []) + (["-DKDA_DEBUG"] if debug else [])
        subprocess.run(command(tmp, extra), check=True)
        os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list:
    """The product library and its bounds-checked twin, compiled side by side."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(2) as ex:
        futs = [ex.submit(build_library, force, False, dbg) for dbg in (False, True)]
        return [f.result() for f in futs]


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
