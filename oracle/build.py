"""Compile the CPU oracle into ``oracle/liboracle.so`` with gcc.

Test infrastructure: the library it builds is loaded only by the tests, the
smoke check and the benchmark's CPU-baseline leg.

``-ffp-contract=off`` keeps every ``a*b + c`` of the oracle a separate
multiply and add (gcc on aarch64 would otherwise fuse them), so the oracle
gives the same bits on x86-64 and Arm hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dspark_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
