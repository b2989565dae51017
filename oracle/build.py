"""Build the CPU oracle (plain C, gcc) into ``oracle/liboracle.so``.

Test infrastructure only: the oracle is compiled so that the test-suite, the
smoke check and the benchmark's CPU-baseline leg can call it.  The product
library never links or loads it.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

# IEEE arithmetic only: no fast-math, no contraction of a*b+c into an FMA,
# no flush-to-zero.
# OpenMP only spreads whole output rows over threads (see fp8_oracle.c).
CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
          "-ffp-contract=off", "-fno-finite-math-only", "-fopenmp", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    subprocess.run(["gcc", *CFLAGS, "-o", LIB, SRC, "-lm"], check=True)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
