"""Compile the CPU oracle (plain C) into a shared library.

Test infrastructure: only the tests, the smoke check and the benchmark's
CPU-baseline leg use the result.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rmsq_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "librmsq_oracle.so")

# No fast-math and no contraction: every rounding in the source is the one
# the definition states.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra", "-pthread"]


def compile_source(src: str, out: str) -> str:
    """Compiles an oracle source file (used by the tests that plant mistakes)."""
    subprocess.run(["gcc", *CFLAGS, "-o", out, src, "-lm"], check=True)
    return out


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
