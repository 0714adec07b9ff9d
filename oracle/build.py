"""Compile the oracle's C sources into oracle/liboracle.so with gcc.

The oracle is test infrastructure: this only builds the checker, it does
not put the oracle on any product code path.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ["scan_ref.c", "tile_model.c"]
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, extra_flags: list[str] | None = None, out: str | None = None) -> str:
    """Build the shared library; returns its path.  `extra_flags` and `out`
    exist so a test can build a deliberately broken copy elsewhere."""
    target = out or LIB
    srcs = [os.path.join(HERE, s) for s in SOURCES]
    if not force and out is None and os.path.exists(target):
        newest = max(os.path.getmtime(s) for s in srcs + [__file__])
        if os.path.getmtime(target) >= newest:
            return target
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC",
           *(extra_flags or []), "-o", target, *srcs]
    subprocess.run(cmd, check=True)
    return target


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
