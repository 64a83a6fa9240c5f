"""Builds the oracle's shared library (plain C, gcc, OpenMP).

Test infrastructure: the oracle is compiled here so that the test-suite, the
smoke check and the CPU-baseline leg of the benchmark can load it.  Nothing in
the product library links against it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8kv_oracle.c")
LIB = os.path.join(HERE, "_build", "liboracle.so")


def build(force: bool = False) -> str:
    """Compiles liboracle.so if it is missing or older than its source."""
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    # -ffp-contract=off: no fused multiply-add, so x86 and Arm hosts compute
    # the same fp64 sums; no -ffast-math: the fp32 divide must stay IEEE.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
