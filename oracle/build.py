"""Compile the CPU oracle (test infrastructure) into ``oracle/liboracle_kv4.so``.

Plain gcc, no contraction of float expressions (``-ffp-contract=off``) so the
oracle rounds exactly as its source is written, no fast-math, OpenMP for the
batch entry that times the CPU baseline.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kv4_oracle.c")
LIB = os.path.join(HERE, "liboracle_kv4.so")

CFLAGS = ["-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra", "-fopenmp"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source; return its path."""
    deps = [SRC, os.path.join(HERE, "kv4_oracle.h"), os.path.abspath(__file__)]
    if not force and os.path.exists(LIB):
        if os.path.getmtime(LIB) >= max(os.path.getmtime(d) for d in deps):
            return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
