"""Compile the fp64 CPU oracle (test infrastructure) into oracle/_build/liboracle.so.

Plain gcc, no CUDA. -ffp-contract=off keeps every fp64 multiply and add a
separate correctly rounded operation on every host architecture.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")
SRC = os.path.join(HERE, "oracle.c")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(src: str = SRC, out: str = LIB, extra: list[str] | None = None) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", *CFLAGS, *(extra or []), "-I", HERE, "-o", out + ".tmp", src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    lib_t = os.path.getmtime(LIB)
    return any(os.path.getmtime(os.path.join(HERE, f)) > lib_t for f in ("oracle.c", "oracle.h"))


if __name__ == "__main__":
    print(build(), file=sys.stderr)
