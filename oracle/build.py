"""Build the CPU oracle (test infrastructure) into oracle/liboracle_zero.so.

The oracle is plain C compiled without FMA contraction and without fast-math,
so every `a * b + c` in it is two IEEE roundings, as written.  Only the tests,
the smoke check and the benchmark's CPU-baseline leg load the result.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "zero_oracle.c")
LIB = os.path.join(HERE, "liboracle_zero.so")

CFLAGS = [
    "-O2", "-std=c11", "-fPIC", "-shared",
    "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard",
    "-fno-strict-aliasing", "-fno-semantic-interposition", "-Wall",
]


def build(force: bool = False) -> str:
    """Compile the oracle if the source is newer than the library; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(os.path.join(HERE, "zero_oracle.h"))):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
