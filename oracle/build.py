"""Compile the fp64 CPU oracle into ``oracle/_build/liboracle.so``.

Test infrastructure: the oracle checks the CUDA path and is never part of it.
Built with the host's gcc (x86_64 or aarch64 alike), OpenMP when the compiler
has it, plain IEEE arithmetic (no fast-math, no -march).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "sdv_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle if the source is newer than the library; return its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    deps = [SRC, os.path.join(HERE, "sdv_oracle.h")]
    if not force and os.path.exists(LIB) and all(
            os.path.getmtime(LIB) >= os.path.getmtime(d) for d in deps):
        return LIB
    base = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-Wall", "-o", LIB + ".tmp", SRC]
    for extra in (["-fopenmp"], []):
        r = subprocess.run(base + extra + ["-lm"], capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(LIB + ".tmp", LIB)
            return LIB
    sys.stderr.write(r.stderr)
    raise RuntimeError("oracle build failed")


if __name__ == "__main__":
    print(build(force=True))
