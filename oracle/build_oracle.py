"""Compile the CPU oracle (test infrastructure only) into oracle/liboracle.so.

Plain gcc, no fast-math and no contraction of a*b+c into fused multiply-adds,
so the fp64 arithmetic is the same on x86-64 and on AArch64 hosts.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gemm_relu_oracle.c")
ATTENTION_SRC = os.path.join(HERE, "attention_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(src=SRC, out=LIB, extra_flags=(), attention_src=ATTENTION_SRC):
    """Compile the GEMM + ReLU oracle `src` and the attention oracle
    `attention_src` into the shared library `out`; return its path."""
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-shared", "-fPIC", *extra_flags, "-o", out, src, attention_src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def needs_build(src=SRC, out=LIB):
    return (not os.path.exists(out)) or any(
        os.path.getmtime(out) < os.path.getmtime(f) for f in (src, ATTENTION_SRC))


if __name__ == "__main__":
    print(build())
