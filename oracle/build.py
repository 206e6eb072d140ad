"""Compile the CPU oracle (``poetx_oracle.c``) into ``liboracle.so``.

TEST INFRASTRUCTURE ONLY: the oracle is the slow double-precision statement
of the method that the GPU library is checked against.  Building it is part of
``__graft_entry__.build()``; the tests build it on demand when it is missing.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "poetx_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

# -ffp-contract=off keeps every multiply and add a separately rounded IEEE
# double operation, so the oracle's results do not depend on FMA contraction.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-lm"]


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *CFLAGS[:-1], SRC, "-o", tmp, CFLAGS[-1]]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
