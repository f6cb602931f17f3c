"""Compile the CPU oracle (test infrastructure) into oracle/libmoe_oracle.so."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "libmoe_oracle.so")

# No fast-math and no FMA contraction: the fp32 activation quantiser must be
# plain IEEE division followed by rintf.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-pthread"]


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        subprocess.check_call(["gcc", *CFLAGS, SRC, "-o", LIB, "-lm"])
    return LIB


if __name__ == "__main__":
    print(build(force=True))
