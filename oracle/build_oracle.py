"""Compile the CPU oracle (plain C) into oracle/libdt_oracle.so.

Test infrastructure only: the library this builds is loaded by the tests, the
smoke check and the benchmark's CPU-baseline leg, never by the product path.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dt_oracle.c")
LIB = os.path.join(HERE, "libdt_oracle.so")

# -std=c11 and -ffp-contract=off: IEEE binary32 arithmetic exactly as written,
# no fused multiply-add on any host (gcc contracts by default on aarch64).
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-pthread", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
