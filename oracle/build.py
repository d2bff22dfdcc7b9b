"""Compile the float64 CPU oracle (test infrastructure) into a shared library.

Plain gcc, no CUDA: ``python -m oracle.build`` or ``build()``.  The library is
written to ``oracle/_build/liboracle.so``; ``build(out, src)`` can compile another
source (the mutation tests use it to compile deliberately broken copies).
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT = os.path.join(HERE, "_build", "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
          "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(out: str = OUT, src: str = SRC, quiet: bool = True) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, src, "-o", tmp, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{' '.join(cmd)}\n{res.stderr}")
    if not quiet and res.stderr:
        print(res.stderr)
    os.replace(tmp, out)
    return out


def needs_build(out: str = OUT, src: str = SRC) -> bool:
    return (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)


if __name__ == "__main__":
    print(build(quiet=False))
