"""Build the fp8bs shared library in-tree for sm_103a.

    python -m fp8_fine_grained_15_b300.build [--verbose]

Produces ``fp8_fine_grained_15_b300/libfp8bs.so`` from ``csrc/fp8bs.cu`` (one
translation unit that includes the kernel headers).  The CUDA runtime is linked
statically; the driver's tensor-map encoder is fetched at run time, so the
library loads on a machine without a GPU driver.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libfp8bs.so")
SOURCES = [os.path.join(CSRC, "fp8bs.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "quant_kernels.cuh", "gemm_pair_kernel.cuh",
                                                  "gemm_mx_kernel.cuh", "gemm_kernel.cuh")] + \
    [os.path.join(ROOT, "include", "fp8bs.h")]

NVCC_FLAGS = [
    "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "--expt-relaxed-constexpr", "-cudart", "static",
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [nvcc(), *NVCC_FLAGS, *(["-Xptxas", "-v"] if verbose else []), "-o", tmp, *SOURCES]
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose="--verbose" in sys.argv)
    print(LIB)
