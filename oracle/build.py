"""Compile the C part of the oracle with the host compiler (test infrastructure).

Builds ``oracle/liboracle_w4.so`` from ``w4_ref.c`` with plain IEEE
arithmetic (no fast-math, no FMA contraction) and OpenMP over output columns.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "w4_ref.c")
LIB = os.path.join(HERE, "liboracle_w4.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cmd = [
        os.environ.get("CC", "gcc"), "-O2", "-fno-fast-math", "-ffp-contract=off",
        "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", LIB + ".tmp", SRC, "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
