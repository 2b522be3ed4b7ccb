"""Compile the oracle (plain C) into a shared library with gcc.

The oracle is test infrastructure: building it here does not make it part of the product path.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")
SOURCE = os.path.join(HERE, "oracle.c")

# -ffp-contract=off keeps every multiply and add a separate IEEE operation, as written.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(source: str = SOURCE, out: str = LIB_PATH, extra_flags=()) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, *extra_flags, source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def is_stale(out: str = LIB_PATH, source: str = SOURCE) -> bool:
    return not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(source)


if __name__ == "__main__":
    print(build())
    sys.exit(0)
