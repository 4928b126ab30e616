"""Compile the oracle (test infrastructure) into oracle/libkvq_oracle.so with gcc.

The oracle is plain C, single-threaded, built without fast-math and without
floating-point contraction so that each fp32 operation rounds exactly once.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kvq_oracle.c")
LIB = os.path.join(HERE, "libkvq_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(src: str = SRC, out: str = LIB, extra_flags: list[str] | None = None, force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source; return its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", *CFLAGS, *(extra_flags or []), src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
