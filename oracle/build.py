"""Compile the CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain g++ with floating-point contraction off, so every rounding happens where
oracle.cpp writes it.  Works the same on x86-64 and aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.cpp")
LIB = os.path.join(HERE, "liboracle.so")
FLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def compile_source(src: str, out: str) -> str:
    """Compile one C++ source with the oracle's flags into the shared library out."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["g++", *FLAGS, "-o", tmp, src], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    return compile_source(SRC, LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
