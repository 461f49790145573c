"""Build the CPU oracle's shared library (TEST INFRASTRUCTURE ONLY).

Compiles ``muon_oracle.c`` with gcc into ``liboracle_muon.so`` beside it.
``-ffp-contract=off`` is required: the oracle's rounding points are part of
its definition, and a compiler-contracted multiply-add would change them.
OpenMP only splits output rows across threads; every output element is still
summed by one thread in a fixed order, so results do not depend on it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "muon_oracle.c")
LIB = os.path.join(HERE, "liboracle_muon.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-O3", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-shared", "-fPIC", SRC, "-o", LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # no OpenMP runtime: single-threaded build, same results
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
