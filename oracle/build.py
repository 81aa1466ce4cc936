"""Compile the CPU oracle (oracle.c) into oracle/_build/liboracle.so with gcc.

Test infrastructure only: the tests, the smoke check and the benchmark's
CPU-baseline leg load the result; the product library never does.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-Wall", "-o", tmp, SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)  # no OpenMP runtime: single thread
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
