"""Compile the plain-C oracle into oracle/_build/liboracle.so.

Test infrastructure only: the oracle is the CPU definition the CUDA path is
checked against.  gcc, -O2, no FMA contraction, no fast-math, no -march, so
the result is the same IEEE fp32 arithmetic on x86_64 and aarch64.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = [os.path.join(HERE, "oracle.c")]
HDR = [os.path.join(HERE, "oracle.h")]
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fno-strict-aliasing",
          "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra"]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in SRC + HDR)


def build(force: bool = False) -> str:
    if force or stale():
        os.makedirs(OUT_DIR, exist_ok=True)
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, *SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
