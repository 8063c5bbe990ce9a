"""Compile the fp64 CPU oracle (oracle.c) into oracle/_build/liboracle.so.

Test infrastructure: the library is loaded by the test suite, the smoke
check and the benchmark's CPU-baseline leg only.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")
SRC = os.path.join(HERE, "oracle.c")


def build(force: bool = False) -> str:
    """Build the oracle library if missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".%d.tmp" % os.getpid()
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-Wall",
            "-shared", "-fPIC", SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # a host without libgomp still gets a (single-threaded) oracle
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
