"""Builds libbfp8.so (the C-ABI library) in-tree with nvcc for sm_103a."""

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libbfp8.so")
SOURCES = [os.path.join(HERE, "csrc", "api.cu")]
DEPS = SOURCES + [os.path.join(HERE, "csrc", f) for f in ("common.cuh", "quant.cuh", "gemm.cuh", "gemm_mx.cuh")] + [
    os.path.join(ROOT, "include", "bfp8.h")]

NVCC_FLAGS = [
    "-O3", "-std=c++17",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo",
    "-Xcompiler", "-fPIC", "-shared",
    "-cudart", "static",
    "-Xptxas", "-v",
]


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force=False, verbose=False):
    """Compile the library unless it is newer than every source.

    The ptxas resource report (registers, spills, shared memory per kernel)
    is written next to the library as ``libbfp8.ptxas.txt``.
    """
    if not force and up_to_date():
        return LIB
    cmd = [nvcc()] + NVCC_FLAGS + ["-I", os.path.join(ROOT, "include"), "-o", LIB] + SOURCES
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(HERE, "libbfp8.ptxas.txt"), "w") as f:
        f.write(r.stdout + r.stderr)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed building libbfp8.so")
    if verbose:
        print(r.stdout + r.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
