"""Compile the oracle's C source into oracle/_build/liboracle.so with gcc.

Test infrastructure: the product library never loads the result.  Run as a
script (``python oracle/build.py``) or call ``build()``.  OpenMP is used when
the host compiler supports it (independent pages on several host threads);
otherwise the same source builds single-threaded.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "puzzlekv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def _stale() -> bool:
    return (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def build(force: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", SRC, "-o", tmp, "-lm"]
    r = subprocess.run(base[:2] + ["-fopenmp"] + base[2:], capture_output=True, text=True)
    if r.returncode != 0:
        r = subprocess.run(base, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
