"""Compile the CPU oracle into oracle/libmoe_oracle.so (host compiler, OpenMP).

Test infrastructure only: the oracle is plain C++17 built without fast-math, so
every sum is evaluated in the order its loop writes it.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = ["numbers.cpp", "router.cpp", "capacity.cpp", "experts.cpp", "combine.cpp",
           "layer.cpp"]
HEADERS = ["moe_oracle.h", "internal.hpp"]
LIB = os.path.join(HERE, "libmoe_oracle.so")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(os.path.join(HERE, f)) > t for f in SOURCES + HEADERS)


def build(force: bool = False) -> str:
    if not force and not _stale():
        return LIB
    cxx = os.environ.get("CXX", "g++")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cxx, "-std=c++17", "-O2", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp] + \
        [os.path.join(HERE, s) for s in SOURCES]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
