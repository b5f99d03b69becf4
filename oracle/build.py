"""Compile the CPU oracle (ep_oracle.c) into a shared library beside it.

Test infrastructure: the oracle is a checker, never part of the product path.
Plain gcc, no fast-math and no floating-point contraction, so that every
float operation in the oracle is one IEEE-754 binary32 operation.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ep_oracle.c")
LIB = os.path.join(HERE, "liboracle_ep.so")
CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-fno-finite-math-only", "-Wall", "-Wextra"]


def build_oracle(force: bool = False) -> str:
    """Build liboracle_ep.so if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
