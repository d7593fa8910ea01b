"""Compile the CPU oracle (plain C, gcc) into oracle/lib/liboracle.so.

Test infrastructure: building the oracle is part of building the tests,
not of the product path. OpenMP is used when the compiler supports it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ("gdn_oracle.c", "mamba2_oracle.c")
HEADERS = ("gdn_oracle.h", "mamba2_oracle.h")
OUT = os.path.join(HERE, "lib", "liboracle.so")


def build(force: bool = False, src_dir: str = HERE, out: str = OUT) -> str:
    """Compile the oracle sources in src_dir into out (by default this package's own library; the
    planted-mistake tests build altered copies elsewhere)."""
    srcs = [os.path.join(src_dir, f) for f in SOURCES]
    hdrs = [os.path.join(src_dir, f) for f in HEADERS]
    os.makedirs(os.path.dirname(out), exist_ok=True)
    newest = max(os.path.getmtime(f) for f in srcs + hdrs + [__file__])
    if not force and os.path.exists(out) and os.path.getmtime(out) >= newest:
        return out
    base = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
            "-Wall", "-Wextra", "-D_GNU_SOURCE", *srcs, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
