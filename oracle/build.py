"""Compile the CPU oracle into ``oracle/liboracle.so`` (plain C11, gcc).

TEST INFRASTRUCTURE: the oracle is the checker of the CUDA path, not part of it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "sp24_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

# -ffp-contract=off: no fused multiply-add contraction, so every fp32
# operation rounds on its own on x86-64 and aarch64 alike.
BASE_FLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
              "-fno-fast-math", "-Wall"]


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc"] + BASE_FLAGS + ["-fopenmp", SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:  # no OpenMP runtime: build single-threaded
        cmd = ["gcc"] + BASE_FLAGS + [SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
