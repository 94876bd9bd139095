"""Build the C-ABI shared library libgemm_f16.so in-tree (``_build/``).

One translation unit, one ``-gencode`` (sm_103a), shared cudart; nvcc
cross-compiles it on a machine without a GPU.
"""
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libgemm_f16.so")
SOURCES = [os.path.join(CSRC, "gemm_api.cu")]
DEPS = SOURCES + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(INCLUDE, "gemm_f16.h")]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
    "-I" + INCLUDE, "-I" + CSRC,
]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in DEPS)


def build(force=False, verbose_ptxas=False):
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and not _stale():
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [NVCC, *FLAGS, *(["-Xptxas", "-v"] if verbose_ptxas else []), "-o", tmp, *SOURCES]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
