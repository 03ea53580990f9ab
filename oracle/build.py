"""Builds the CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc, no CUDA: -O2 for speed, -ffp-contract=off so that no multiply-add
is fused and every fp32 step rounds exactly as written in the source.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gs_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC),
                                             os.path.getmtime(os.path.join(HERE, "gs_oracle.h")))):
        return LIB
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-D_DEFAULT_SOURCE", SRC, "-o", LIB + ".tmp", "-lm", "-lpthread"]
    subprocess.check_call(cmd)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
