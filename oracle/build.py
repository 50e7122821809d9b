"""Compile the CPU oracle (plain C) into oracle/libbi_oracle.so with gcc.

Test infrastructure: the library built here is loaded only by the tests, the
smoke check and the benchmark's CPU-baseline leg.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "bi_oracle.c")
LIB = os.path.join(HERE, "libbi_oracle.so")


def build(force: bool = False) -> str:
    """Build the oracle shared library if it is missing or older than its source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(
        os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "bi_oracle.h"))
    ):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [
        os.environ.get("CC", "gcc"), "-O2", "-std=c11", "-fPIC", "-shared",
        "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
        SRC, "-o", tmp, "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
