"""Compile the oracle's C source into ``oracle/liboracle.so`` (gcc, fp64, OpenMP).

Building the checker is not using it: the product path never loads this
library.  Plain C99, no architecture flags, so the same source builds on x86-64
and on aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fno-fast-math", SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        # a toolchain without libgomp still builds a correct single-threaded oracle
        subprocess.run(base, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
