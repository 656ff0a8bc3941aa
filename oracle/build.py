"""Compile the CPU oracle (plain C) into oracle/_build/libmq_oracle.so.

Test infrastructure: builds the checker, never the product.  Flags keep the
fp32 steps of the q8_0 quantizer exact IEEE (no contraction into FMA, no
fast-math).  Plain C99 that builds the same on x86_64 and aarch64.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mq_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmq_oracle.so")

CFLAGS = ["-std=c99", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def needs_build() -> bool:
    return (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    if force or needs_build():
        os.makedirs(OUT_DIR, exist_ok=True)
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
