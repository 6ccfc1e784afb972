"""Compile the fp64 CPU oracle (oracle.c) into a shared library with gcc.

TEST INFRASTRUCTURE: the library this builds is loaded only by the tests, the
smoke check and the benchmark's CPU-baseline leg.

Portable C (builds the same on x86_64 and aarch64): no -march=native, no
-ffast-math (IEEE semantics for exp/log and the -inf conventions).
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def compile_oracle(src: str = SRC, out: str = LIB, werror: bool = True) -> str:
    """Compile `src` to the shared library `out`; returns `out`."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra"]
    cmd += ["-Werror"] if werror else ["-w"]
    cmd += [src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    """Build liboracle.so next to oracle.c unless it is newer than the source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    return compile_oracle()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
