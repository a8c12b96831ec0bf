"""Compile the CPU oracle (test infrastructure) into oracle/_liboracle.so.

Plain gcc, fp64, OpenMP when the compiler has it.  ``-ffp-contract=off`` keeps
gcc from fusing multiply-adds (aarch64 gcc fuses by default), so the oracle
gives the same bits on x86-64 and on Arm hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkv_oracle.c")
LIB = os.path.join(HERE, "_liboracle.so")


def build(verbose: bool = False, force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", SRC, "-o", LIB + ".tmp", "-lm"]
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(LIB + ".tmp", LIB)
            return LIB
        if verbose:
            print(r.stderr, file=sys.stderr)
    raise RuntimeError("oracle build failed:\n" + r.stderr)


if __name__ == "__main__":
    print(build(verbose=True, force=True))
