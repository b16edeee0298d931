"""Compile the C++ oracle into oracle/_build/libmoe_oracle.so (plain g++, no GPU).

-ffp-contract=off keeps every fp64 operation a separately rounded IEEE
operation on both x86 and Arm (no fused multiply-add contraction).
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmoe_oracle.so")
SRC = [os.path.join(HERE, "moe_oracle.cpp")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in SRC + [os.path.join(HERE, "moe_oracle.h")])


def build(force: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
           "-o", tmp] + SRC + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
