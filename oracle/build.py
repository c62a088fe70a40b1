"""Build the CPU oracle's shared library (test infrastructure only).

``build()`` compiles ``pq2_oracle.c`` with the host gcc into
``libpq2_oracle.so`` beside it.  Plain C, no fast-math, no FMA contraction,
OpenMP over output rows when the compiler supports it.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pq2_oracle.c")
LIB = os.path.join(HERE, "libpq2_oracle.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", SRC, "-o", LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:6] + ["-fopenmp"] + base[6:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
