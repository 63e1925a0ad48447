"""Build the CPU oracle shared library (oracle/liboracle.so) with the host C compiler.

The oracle is test infrastructure: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` load it; the CUDA library never does.

Flags that matter for exactness: ``-ffp-contract=off`` (no fused multiply-add where the
source writes a separate multiply and add) and no ``-ffast-math`` (IEEE division, gradual
underflow, no flush-to-zero).  No architecture-specific flag is used, so the same source
gives the same results on x86_64 and aarch64.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qz_oracle.c")
HDR = os.path.join(HERE, "qz_oracle.h")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = [
    "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
    "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard",
    "-Wall", "-Wextra", "-Wno-unused-parameter",
]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR, __file__))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile liboracle.so if it is missing or older than its sources; return its path."""
    if force or needs_build():
        cc = os.environ.get("CC", "gcc")
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [cc, *CFLAGS, "-o", tmp, SRC, "-lm"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
