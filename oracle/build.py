"""Build the CPU oracle ``libkivi_ref.so`` with gcc.

Test infrastructure only: the CUDA library never links or loads this.
IEEE single-precision arithmetic is kept literal: no fast-math and no
contraction of a*b+c into a fused multiply-add.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kivi_ref.c")
HDR = os.path.join(HERE, "kivi_ref.h")
LIB = os.path.join(HERE, "libkivi_ref.so")

CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
          "-fno-strict-aliasing", "-Wall", "-fPIC", "-shared"]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    lib_t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > lib_t for p in (SRC, HDR, __file__))


def build(force: bool = False) -> str:
    """Compile the oracle if it is missing or stale; return the library path."""
    if force or needs_build():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
