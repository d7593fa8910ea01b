"""Compile the CPU oracle (plain C, gcc) into oracle/lib/liboracle.so.

Test infrastructure: building the oracle is part of building the tests,
not of the product path. OpenMP is used when the compiler supports it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRCS = [os.path.join(HERE, f) for f in ("gdn_oracle.c", "mamba2_oracle.c")]
HDRS = [os.path.join(HERE, f) for f in ("gdn_oracle.h", "mamba2_oracle.h")]
OUT = os.path.join(HERE, "lib", "liboracle.so")


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    newest = max(os.path.getmtime(f) for f in SRCS + HDRS + [__file__])
    if not force and os.path.exists(OUT) and os.path.getmtime(OUT) >= newest:
        return OUT
    base = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
            "-Wall", "-Wextra", "-D_GNU_SOURCE", *SRCS, "-o", OUT + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(OUT + ".tmp", OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
