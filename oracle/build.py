"""Build the C oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc; OpenMP when the compiler supports it.  The product library never
links or loads this file.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mla_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra", "-Wno-unused-parameter"]
    for extra in (["-fopenmp"], []):
        cmd = base + extra + [SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            if verbose and r.stderr:
                print(r.stderr, file=sys.stderr)
            os.replace(tmp, LIB)
            return LIB
    raise RuntimeError("oracle build failed:\n" + r.stderr)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
