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


def library_path(threaded: bool = False):
    return os.path.join(OUT_DIR, "libhsdp_oracle_mt.so" if threaded else "libhsdp_oracle.so")


def build(cc: str = "gcc", threaded: bool = False) -> str:
    """threaded: a separate build of the same source with -fopenmp, for the
    labelled multi-core CPU baseline. Its pragmas split only loops whose
    iterations write disjoint outputs (ranks, parameters, shard rows), so
    every output element is computed by the same operations in the same
    order as in the single-threaded build (the oracle). Without -fopenmp
    the pragmas are ignored."""
    os.makedirs(OUT_DIR, exist_ok=True)
    out = library_path(threaded)
    tmp = out + f".tmp{os.getpid()}"
    flags = CFLAGS + (["-fopenmp"] if threaded else ["-Wno-unknown-pragmas"])
    subprocess.run([cc, *flags, "-I", HERE, SRC, "-o", tmp], check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build())
    print(build(threaded=True))
