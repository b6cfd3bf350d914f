"""Compile the CPU oracle (plain C99) into oracle/libfp8bs_oracle.so.

Test infrastructure only: the CUDA library never links or loads this.
Flags: -O2 without -ffast-math and with -ffp-contract=off, so every FP32
division and multiply is the IEEE round-to-nearest one the definitions name.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8bs_oracle.c")
LIB = os.path.join(HERE, "libfp8bs_oracle.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC),
                                             os.path.getmtime(os.path.join(HERE, "fp8bs_oracle.h")))):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
           "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
