"""Compiles the C oracle into oracle/liboracle_topk.so (test infrastructure only).

Run as ``python oracle/build.py`` or call :func:`build`.  Only the tests, the
smoke check and the benchmark's CPU-baseline leg load the result.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "topk_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle_topk.so")


def build(source: str = SOURCE, output: str = LIBRARY, extra_flags: tuple[str, ...] = ()) -> str:
    """Compiles ``source`` with gcc into the shared library ``output`` and returns its path."""
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC", "-pthread",
           *extra_flags, source, "-o", output, "-lm"]
    subprocess.run(cmd, check=True)
    return output


def up_to_date(source: str = SOURCE, output: str = LIBRARY) -> bool:
    return os.path.exists(output) and os.path.getmtime(output) >= os.path.getmtime(source)


if __name__ == "__main__":
    print(build())
    sys.exit(0)
