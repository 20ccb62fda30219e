"""Build step of the oracle's shared library (plain C, gcc, OpenMP).  Test infrastructure.

``build()`` compiles ``k3o.c`` into ``libk3o.so`` beside it when the library is missing or
older than its sources, and returns the library path.  No x86- or Arm-specific flags: the
same source builds on both hosts.
"""
from __future__ import annotations

import fcntl
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "libk3o.so")
SOURCES = [os.path.join(_HERE, "k3o.c"), os.path.join(_HERE, "k3o.h")]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in SOURCES)


def build(force: bool = False) -> str:
    if not force and not _stale():
        return LIB
    with open(os.path.join(_HERE, ".build.lock"), "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)
        if force or _stale():
            tmp = LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-std=c99", "-O2", "-fno-fast-math", "-ffp-contract=off", "-Wall",
                   "-Wextra", "-Werror", "-fopenmp", "-fPIC", "-shared",
                   os.path.join(_HERE, "k3o.c"), "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
