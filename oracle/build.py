"""Compile the C oracle into ``oracle/_build/liboracle.so`` with gcc.

Test infrastructure only. Plain ``-O2`` without fast-math flags so that the
fp64 sums keep the order written in the source.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "spmv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False, defines=(), out: str | None = None) -> str:
    """Build the oracle library (skipped when it is newer than the source).
    ``defines`` adds ``-D`` macros; ``out`` overrides the output path."""
    out = out or LIB
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and not defines and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(SRC)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    cmd[1:1] = [f"-D{d}" for d in defines]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
