"""Compile the fp64 CPU oracle (oracle.c) into liboracle.so next to this file.

Test infrastructure only: the oracle checks the CUDA library and times the CPU
baseline; the product path never loads it. Built with plain gcc, OpenMP when
the compiler has it, no fast-math, so that it builds the same way on x86_64 and
aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")


def build(verbose: bool = False) -> str:
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            SOURCE, "-o", LIBRARY, "-lm"]
    attempts = [base[:1] + ["-fopenmp"] + base[1:], base]
    last = None
    for cmd in attempts:
        proc = subprocess.run(cmd, capture_output=True, text=True)
        if proc.returncode == 0:
            if verbose:
                print(" ".join(cmd))
            return LIBRARY
        last = proc
    raise RuntimeError("oracle build failed:\n" + last.stderr)


if __name__ == "__main__":
    print(build(verbose=True))
    sys.exit(0)
