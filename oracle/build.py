"""Builds the CPU oracle's shared library with the host C compiler.

TEST INFRASTRUCTURE ONLY: the library built here is loaded by the tests, the
package smoke check and the benchmark's CPU-baseline leg, never by the
product path.

The flags keep IEEE binary32 semantics: no fast-math, no floating-point
contraction, no target-specific instruction set (the same source builds on
x86-64 and aarch64 and gives the same bits).
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "arx_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared",
          "-ffp-contract=off", "-fno-fast-math", "-fno-unsafe-math-optimizations",
          "-frounding-math", "-pthread", "-Wall", "-Wextra"]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``arx_oracle.c`` into ``_build/liboracle.so`` if it is stale."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [os.environ.get("CC", "gcc"), *CFLAGS, SRC, "-o", tmp]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
