"""Compile the CPU oracle (oracle.c) into oracle/liboracle.so.

Test infrastructure: building the checker is not using it.  Plain gcc,
OpenMP when the compiler has it, no architecture-specific flags, so the same
source builds on the x86 development host and on the Arm GPU host.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
HDR = os.path.join(HERE, "oracle.h")
LIB = os.path.join(HERE, "liboracle.so")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR, __file__))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
            "-Wno-unknown-pragmas", SRC, "-o", LIB + ".tmp", "-lm"]
    last = None
    for extra in (["-fopenmp"], []):
        cmd = base[:1] + extra + base[1:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(LIB + ".tmp", LIB)
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            return LIB
        last = r
    raise RuntimeError("oracle build failed:\n" + (last.stderr if last else ""))


if __name__ == "__main__":
    print(build(force=True, verbose=True))
