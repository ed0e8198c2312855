"""Compile the CPU oracle (oracle/oref.c) into oracle/liboref.so with the host gcc.

Test infrastructure: building the checker is not using it.  The flags keep the
oracle's float arithmetic exactly as written (no contraction into FMA, no
fast-math); OpenMP is used only to split independent rows across host cores
and is dropped if the toolchain lacks it.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oref.c")
LIB = os.path.join(HERE, "liboref.so")

_BASE_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Build liboref.so if it is missing or older than its source; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp"
    cmd = ["gcc", *_BASE_FLAGS, "-fopenmp", SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        cmd = ["gcc", *_BASE_FLAGS, SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
