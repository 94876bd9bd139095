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


def _stale_lib(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in DEPS)


def _compile(lib, extra):
    tmp = lib + ".tmp%d" % os.getpid()
    subprocess.run([NVCC, *FLAGS, *extra, "-o", tmp, *SOURCES], check=True)
    os.replace(tmp, lib)
    return lib


def build(force=False, verbose_ptxas=False):
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and not _stale_lib(LIB):
        return LIB
    return _compile(LIB, ["-Xptxas", "-v"] if verbose_ptxas else [])


# The measurement build with phase stamps in the single-CTA / CTA-pair kernel
# (GEMM_F16_PHASE_TRACE; see gemm_f16_trace_set).  Never loaded by the product.
TRACE_LIB = os.path.join(OUT_DIR, "libgemm_f16_trace.so")


def build_trace(force=False):
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and not _stale_lib(TRACE_LIB):
        return TRACE_LIB
    return _compile(TRACE_LIB, ["-DGEMM_F16_PHASE_TRACE"])


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
