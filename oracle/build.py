"""Compile the C oracle (test infrastructure) into oracle/_build/liboracle.so."""
from __future__ import annotations

import os
import pathlib
import subprocess

HERE = pathlib.Path(__file__).resolve().parent
SRC = HERE / "pkv_oracle.c"
OUT_DIR = HERE / "_build"
LIB = OUT_DIR / "liboracle.so"


def build(force: bool = False) -> pathlib.Path:
    OUT_DIR.mkdir(exist_ok=True)
    if not force and LIB.exists() and LIB.stat().st_mtime >= SRC.stat().st_mtime:
        return LIB
    tmp = OUT_DIR / f"liboracle.{os.getpid()}.so"
    # Plain IEEE arithmetic: no -ffast-math, no contraction of a*b+c into fma.
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", str(tmp), str(SRC), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
