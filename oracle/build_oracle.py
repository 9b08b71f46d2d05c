"""Compile the CPU oracle (test infrastructure only) into oracle/liboracle.so.

Plain gcc, no fast-math and no contraction of a*b+c into fused multiply-adds,
so the fp64 arithmetic is the same on x86-64 and on AArch64 hosts.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gemm_relu_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(src=SRC, out=LIB, extra_flags=()):
    """Compile `src` to the shared library `out` and return its path."""
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-shared", "-fPIC", *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def needs_build(src=SRC, out=LIB):
    return (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)


if __name__ == "__main__":
    print(build())
