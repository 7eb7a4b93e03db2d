"""Builds the fp64 oracle (test infrastructure) with gcc: plx_oracle.c ->
libplx_oracle.so beside it.  Plain C, -O2, no fast-math and no FMA
contraction, so every operation is a correctly rounded IEEE double op."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "plx_oracle.c")
OUT = os.path.join(HERE, "libplx_oracle.so")


def build(verbose: bool = False, src: str = SRC, out: str = OUT) -> str:
    """Compile ``src`` into the shared library ``out`` (atomically replaced)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True))
