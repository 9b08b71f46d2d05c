"""Build libgemmrelu.so in-tree with nvcc for sm_103a (one translation unit)."""
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
SOURCES = [os.path.join(CSRC, "gemm_relu_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("gemm_relu_kernels.cuh", "gemm_relu_splitk.cuh", "gemm_relu_2sm.cuh", "gemm_relu_gemv.cuh", "flash_attention.cuh", "sm103.cuh", "gemm_relu_stage.cuh")] + [
    os.path.join(INCLUDE, "gemm_relu.h"), os.path.join(INCLUDE, "flash_attention.h")]
LIB = os.path.join(PKG, "libgemmrelu.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
    "-cudart", "static",
]


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def needs_build():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in DEPS)


def build(verbose=False, extra=()):
    cmd = [nvcc(), *NVCC_FLAGS, f"-I{INCLUDE}", f"-I{CSRC}", *extra, "-o", LIB, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    return LIB


if __name__ == "__main__":
    build(verbose="-v" in sys.argv)
