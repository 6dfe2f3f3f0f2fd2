"""Compile the C oracle into ``oracle/liboracle.so`` (gcc, no CUDA).

The oracle is test infrastructure: it is compiled only so that the test-suite,
the smoke check and the benchmark's CPU-baseline leg can load it.  Plain
``-O2`` and no target-specific flags, so the same source builds and gives
the same results on x86-64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def compile_to(src: str, out: str, quiet: bool = False) -> None:
    """Compile one C source of the oracle into the shared library ``out``
    (``quiet``: keep the compiler's warnings out of the output)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-Wextra", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=quiet)


def build(force: bool = False) -> str:
    """Build liboracle.so if missing or older than oracle.c; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    compile_to(SRC, tmp)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
