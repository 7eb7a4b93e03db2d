"""Builds libplx.so (the CUDA kernels + C ABI) in-tree with nvcc for sm_103a.

    python -m parameterized_local_linear_02_b300.build

The library links the CUDA runtime statically and resolves the driver's
tensor-map encoder at run time, so it loads on a host without a GPU (the
symbols can be inspected there; compute calls need a B300)."""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libplx.so")
# the same sources with -DPLX_DEBUG: bounds checks that record PLX_ERR_BOUNDS
# and skip the access (for tests; not the product library)
DEBUG_LIB = os.path.join(PKG, "libplx_debug.so")

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
              "-Xcompiler", "-fPIC", "-shared", "-Xptxas", "-warn-spills"]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in sources())


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    """Compile csrc/plx.cu into libplx.so (or, with ``debug``, libplx_debug.so
    with -DPLX_DEBUG) next to this file (atomic replace)."""
    lib = DEBUG_LIB if debug else LIB
    if not force and not stale(lib):
        return lib
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *NVCC_FLAGS, *(["-DPLX_DEBUG"] if debug else []), f"-I{INCLUDE}", f"-I{CSRC}", "-o", tmp,
           os.path.join(CSRC, "plx.cu")]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv, debug="--debug" in sys.argv))
