"""Build the oracle's shared library (oracle/liboracle.so) with the host C++
compiler.

Test infrastructure only: the oracle is compiled so that tests and the
bench's CPU-baseline leg can call it; the product path never loads it.

Flags: -O2 -ffp-contract=off (no contracted multiply-adds, which gcc would
otherwise emit on aarch64), no -ffast-math, no -march=native.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    # a test may point the oracle at another build of it (the mutation
    # check of the pins builds copies of oracle.cpp with planted mistakes)
    override = os.environ.get("ORACLE_LIB")
    if override:
        return override
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cxx = os.environ.get("CXX", "g++")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cxx, "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
