"""Build the fp64 CPU oracle (plain C + OpenMP) into oracle/_build/.

Test infrastructure: compiled by ``__graft_entry__.build()`` and on demand by the
tests; the product library never uses it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "longstraw_oracle.c")
SRCS = [SRC, os.path.join(HERE, "gdn_oracle.c"), os.path.join(HERE, "mla_oracle.c")]
HDR = os.path.join(HERE, "longstraw_oracle.h")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "liblongstraw_oracle.so")


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in (*SRCS, HDR, __file__))


def build(force: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-Wno-unused-parameter", "-o", tmp, *SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
