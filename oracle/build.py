"""Compile the fp64 CPU oracle (test infrastructure) into oracle/libmoe_oracle.so.

Plain C99, -O2, no fast-math; OpenMP over tokens when the compiler has it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "libmoe_oracle.so")


def build(force: bool = False) -> str:
    hdr = os.path.join(HERE, "moe_oracle.h")
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC), os.path.getmtime(hdr))):
        return LIB
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-std=c99", "-O2", "-fno-fast-math", "-fPIC", "-shared", "-Wall", "-Wextra"]
    tmp = LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", SRC, "-o", tmp, "-lm"], check=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
