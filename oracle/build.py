"""Compile the C oracle into ``oracle/liboracle.so`` (test infrastructure).

The oracle is the checker the CUDA path is compared against; only the tests,
the smoke check and the benchmark's CPU-baseline leg use it.  Contraction is
switched off so every binary32 operation is rounded on its own, in the order
the source writes it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "asr_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
          "-fno-unsafe-math-optimizations", "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
