"""Compile the FP64 CPU oracle (``pkv_oracle.c``) into ``liboracle.so``.

Test infrastructure: the oracle is built so that the test suite, the smoke
check and the benchmark's CPU-baseline leg can call it.  Plain gcc, C11,
``-ffp-contract=off`` so no multiply-add is fused and x86-64 and AArch64 give
the same bits.  No ``-march=native`` and no ``-ffast-math``.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkv_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, verbose: bool = False) -> str:
    """Build ``liboracle.so`` next to the source if it is missing or stale."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [
        os.environ.get("CC", "gcc"), "-std=c11", "-O2", "-fPIC", "-shared",
        "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
        "-o", tmp, SRC, "-lm",
    ]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
