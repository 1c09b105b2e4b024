"""Builds the CPU oracle (plain C) into oracle/liboq8.so.

Test infrastructure: building the checker is not using it.  Portable flags only (the
library is built on x86-64 and on aarch64 hosts); -ffp-contract=off keeps the compiler
from fusing a*b+c, so both hosts round every step the same way.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "q8_oracle.c")
LIB = os.path.join(HERE, "liboq8.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-pthread", SRC, "-o", LIB + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
