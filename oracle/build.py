"""Builds the CPU oracles (plain C): oracle/liboq8.so (the Q8_0 linear layer),
oracle/libokv3.so (the 3-bit KV-cache codec) and oracle/libobsa.so (block-sparse
attention).

Test infrastructure: building the checker is not using it.  Portable flags only (the
libraries are built on x86-64 and on aarch64 hosts); -ffp-contract=off keeps the compiler
from fusing a*b+c, so both hosts round every step the same way.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "q8_oracle.c")
LIB = os.path.join(HERE, "liboq8.so")
KV3_SRC = os.path.join(HERE, "kv3_oracle.c")
KV3_LIB = os.path.join(HERE, "libokv3.so")
BSA_SRC = os.path.join(HERE, "bsa_oracle.c")
BSA_LIB = os.path.join(HERE, "libobsa.so")


def _build_one(src: str, lib: str, force: bool) -> str:
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(src):
        return lib
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           "-pthread", src, "-o", lib + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(lib + ".tmp", lib)
    return lib


def build(force: bool = False) -> str:
    return _build_one(SRC, LIB, force)


def build_kv3(force: bool = False) -> str:
    return _build_one(KV3_SRC, KV3_LIB, force)


def build_bsa(force: bool = False) -> str:
    return _build_one(BSA_SRC, BSA_LIB, force)


if __name__ == "__main__":
    f = "--force" in sys.argv
    print(build(force=f), build_kv3(force=f), build_bsa(force=f))
