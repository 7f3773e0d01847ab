"""Build libkivi_gb300.so in-tree with nvcc for sm_103a (GB300).

Usage: python -m kivi_kv_cache_gb300.build [--force]

Each CUDA translation unit is compiled in parallel, then linked into a shared
library with the CUDA runtime linked statically, so the library loads on any
machine with the CUDA driver (and on a machine without a GPU, where only the
host-side entry points work). No fast-math: every fp32 step of the quantizer
must round like IEEE binary32.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkivi_gb300.so")
SOURCES = ["kivi_api.cu", "flush.cu", "dequant.cu", "decode_mma.cu", "decode_mma_f16s.cu", "decode_mma_d64.cu",
           "decode_mma_d256.cu", "decode_mma_d256_f16s.cu", "decode_pair.cu", "residual.cu", "decode_noalloc.cu",
           "kivi_cache.cu"]
HEADERS = ["kivi_device.cuh", "kivi_launch.h", "decode_merge.cuh", "decode_common.cuh", "decode_mma.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _newest_input() -> float:
    paths = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    paths.append(os.path.join(ROOT, "include", "kivi.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(OBJ, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(OBJ, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc(), *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".%d.tmp" % os.getpid()
    cmd = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-cudart", "static",
           "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
