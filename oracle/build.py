"""Compile the CPU oracle (``oracle.c``) into ``liboracle.so`` beside it.

Test infrastructure: the oracle is the yardstick for the CUDA library and is
never part of the product path.  Plain gcc, no fast-math and no floating-point
contraction, so every binary32 operation in the C source is the one executed
(gcc contracts a*b+c into an FMA by default on aarch64 unless told not to).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build liboracle.so if it is missing or older than its source; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [os.environ.get("CC", "gcc")] + CFLAGS + [SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
