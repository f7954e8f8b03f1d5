"""Compiles the fp64 CPU oracle (kda_oracle.c) into a shared library.

TEST INFRASTRUCTURE ONLY: the library is loaded by ``oracle`` for the tests,
the smoke check and the CPU-baseline leg of the benchmark.  Plain gcc, no
vector extensions and no FMA contraction, so that x86_64 and aarch64 hosts
evaluate the same expression tree.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kda_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libkda_oracle.so")


def build(force: bool = False) -> str:
    """Builds ``_build/libkda_oracle.so`` if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
