"""Compile the C oracle (test infrastructure) into ``oracle/libep_oracle.so``.

The oracle is built with ``-ffp-contract=off`` so that every fp32 product and
sum in its combine fold rounds on its own; no other optimisation changes what
it computes.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ep_oracle.c")
LIB = os.path.join(HERE, "libep_oracle.so")
LIB_OMP = os.path.join(HERE, "libep_oracle_omp.so")


def build(force: bool = False, verbose: bool = False, openmp: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source; return its
    path. ``openmp``: the same source built with -fopenmp (for timing on all host
    cores; identical results)."""
    lib = LIB_OMP if openmp else LIB
    if (not force and os.path.exists(lib)
            and os.path.getmtime(lib) >= os.path.getmtime(SRC)):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-Wall",
           *(["-fopenmp"] if openmp else ["-Wno-unknown-pragmas"]), "-fPIC", "-shared", "-o", tmp, SRC]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
