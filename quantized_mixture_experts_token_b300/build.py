"""Build libmoeq.so (CUDA, sm_103a) in-tree with nvcc."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmoeq.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "--expt-relaxed-constexpr",
    "-cudart", "static",
]


PEAKS_LIB = os.path.join(HERE, "libmoeq_peaks.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cuh")) and f != "peaks.cu")


def _build_one(src, lib, deps, force, verbose):
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= max(os.path.getmtime(d) for d in deps):
        return lib
    cmd = [NVCC, *FLAGS, src, "-o", lib + ".tmp"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(lib + ".tmp", lib)
    return lib


def build(force: bool = False, verbose: bool = False) -> str:
    """libmoeq.so (the layer) and libmoeq_peaks.so (its int8 peak microbenchmark)."""
    inc = os.path.join(ROOT, "include")
    _build_one(os.path.join(CSRC, "moeq.cu"), LIB, sources() + [os.path.join(inc, "moeq.h"), __file__], force,
               verbose)
    peaks_src = os.path.join(CSRC, "peaks.cu")
    _build_one(peaks_src, PEAKS_LIB, [peaks_src, os.path.join(inc, "moeq_peaks.h"), __file__], force, verbose)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force=True, verbose="-v" in sys.argv))
