"""Compile the CPU oracle (oracle.c) into liboracle.so with gcc.

Test infrastructure: the library it builds is only loaded by the tests, the smoke
check and the benchmark's CPU-baseline leg.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
HDR = os.path.join(HERE, "oracle.h")
LIB = os.path.join(HERE, "liboracle.so")


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR, __file__))


def build(force: bool = False) -> str:
    """Build liboracle.so if it is missing or older than its sources; return its path."""
    if force or stale():
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
