"""Builds the CPU oracle (test infrastructure) into oracle/_build/.

Plain C11, -O2, no FMA contraction and no fast-math, so each float operation
in the source is one IEEE binary32 operation with subnormals kept. Portable
C only (no intrinsics, no -march), so it builds the same on x86-64 and
aarch64 hosts.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "hsdp_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra", "-Werror"]


def library_path():
    return os.path.join(OUT_DIR, "libhsdp_oracle.so")


def build(cc: str = "gcc") -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    out = library_path()
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run([cc, *CFLAGS, "-I", HERE, SRC, "-o", tmp], check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build())
