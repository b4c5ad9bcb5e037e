"""Compile the fp64 CPU oracle (plain C) into ``oracle/libtpmlp_oracle.so``.

Test infrastructure: the oracle is built so the tests, the smoke check and
the benchmark's CPU-baseline leg can call it; the product never does.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "tpmlp_oracle.c")
LIB = os.path.join(HERE, "libtpmlp_oracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    base = ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp", "-lm"]
    # OpenMP splits independent outputs across host cores; fall back to a
    # serial build if the compiler lacks it.
    for extra in (["-fopenmp"], []):
        cmd = base[:5] + extra + base[5:]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode == 0:
            os.replace(LIB + ".tmp", LIB)
            return LIB
    raise RuntimeError("oracle build failed")


if __name__ == "__main__":
    print(build(force=True, verbose=True))
