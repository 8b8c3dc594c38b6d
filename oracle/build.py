"""Compile the FP64 oracle (plain C + OpenMP) into a shared library.

TEST INFRASTRUCTURE ONLY: the oracle is built so that tests, the smoke check
and the bench's CPU-baseline leg can run it; nothing on the product path
loads it.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "msa_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Build ``oracle/_build/liboracle.so`` if it is missing or stale."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    build_from(SRC, LIB)
    return LIB


def build_from(src: str, lib: str, extra=()) -> str:
    """Compile ``src`` into ``lib`` (also used to build planted-mistake copies
    of the oracle in the pin tests)."""
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", *extra, src, "-o", tmp,
           "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True))
