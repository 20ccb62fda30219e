"""Build step of the device twin of the synthetic-input generator (``libsynth_dev.so``)."""
from __future__ import annotations

import fcntl
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "libsynth_dev.so")
SRC = os.path.join(_HERE, "synth_dev.cu")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _stale() -> bool:
    return not os.path.exists(LIB) or os.path.getmtime(SRC) > os.path.getmtime(LIB)


def build(force: bool = False) -> str:
    if not force and not _stale():
        return LIB
    with open(os.path.join(_HERE, ".build.lock"), "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)
        if force or _stale():
            tmp = LIB + f".tmp{os.getpid()}"
            cmd = [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                   "-Xcompiler", "-fPIC", SRC, "-o", tmp]
            subprocess.run(cmd, check=True)
            os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
