"""Compile the C oracle into ``oracle/liboracle.so``.

Test infrastructure: the oracle is built so the tests, the smoke check and the
benchmark's CPU-baseline leg can load it; nothing in the product path uses it.

The flags matter: ``-ffp-contract=off`` keeps every fp32 statement of the
oracle a single IEEE operation (no fused multiply-add), and no fast-math flag
is given, so libm and the rounding mode behave as the C standard says.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "maskllm_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build liboracle.so if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
