"""Compile the fp64 CPU oracle into ``oracle/liboal_oracle.so``.

Test infrastructure: the oracle is the correctness reference for the CUDA
library and the timed CPU baseline; no product code path loads it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oal_oracle.c")
LIB = os.path.join(HERE, "liboal_oracle.so")


def build(force: bool = False) -> str:
    """Build the oracle shared library if it is missing or stale; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-std=c11",
           "-Wall", "-Wextra", "-shared", "-fPIC", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
