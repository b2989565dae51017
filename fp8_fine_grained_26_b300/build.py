"""Build ``libfp8bs.so`` (the C-ABI library) in-tree with nvcc for sm_103a."""
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libfp8bs.so")
SOURCES = [os.path.join(CSRC, "fp8bs.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("ptx.cuh", "common.cuh", "quant.cuh", "gemm.cuh")] + \
    [os.path.join(ROOT, "include", "fp8bs.h")]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
# IEEE division and fp32 subnormals are part of the quantiser's contract:
# no fast-math, no flush-to-zero.
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
         "-shared", "-Xcompiler", "-fPIC", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
         "-fmad=true", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in SOURCES + HEADERS)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and not _stale():
        return LIB
    cmd = [NVCC, *FLAGS, "-o", LIB, *SOURCES]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="-v" in sys.argv))
