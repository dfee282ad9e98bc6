"""Compile the fp64 C oracle into ``oracle/liboracle.so`` (gcc, OpenMP).

Test infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline leg load the result; the product library never does.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdn_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, cc: str = "gcc") -> str:
    """Build the oracle if the library is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    # -ffp-contract=off: plain IEEE double evaluation, the same on x86 and Arm.
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
