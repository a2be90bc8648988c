"""Builds the C-ABI library ``lib/libhsdp_fsdp.so`` in-tree.

Four translation units compiled in parallel and linked with nvcc:
  * csrc/fsdp_kernels.cu -- the sm_103a kernels (nvcc, one -gencode)
  * csrc/fsdp_bulk.cu    -- the bulk-fed fused reduce of a capped grid
  * csrc/fsdp_noalloc.cu -- the allocation-free fused gradient sync
  * csrc/fsdp_capi.cpp   -- plan, bindings and entry points (host C++)
No fast-math, no FMA contraction, no flush-to-zero: the kernels' additions,
divisions and conversions are single IEEE operations.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(HERE, "lib")
LIB_NAME = "libhsdp_fsdp.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-Wall", "-ftz=false",
              "-prec-div=true", "-prec-sqrt=true", "-fmad=false", "--expt-relaxed-constexpr"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-Wextra"]


def cuda_home():
    for c in [os.environ.get("CUDA_HOME"), "/usr/local/cuda"]:
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def library_path():
    return os.path.join(LIB_DIR, LIB_NAME)


def build(verbose: bool = False, extra_nvcc=()) -> str:
    cuda = cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(LIB_DIR, exist_ok=True)
    inc = ["-I", INCLUDE, "-I", CSRC]
    tag = str(os.getpid())
    obj_k = os.path.join(LIB_DIR, f"fsdp_kernels.{tag}.o")
    obj_n = os.path.join(LIB_DIR, f"fsdp_noalloc.{tag}.o")
    obj_b = os.path.join(LIB_DIR, f"fsdp_bulk.{tag}.o")
    obj_c = os.path.join(LIB_DIR, f"fsdp_capi.{tag}.o")
    jobs = [
        [nvcc, *ARCH, *NVCC_FLAGS, *extra_nvcc, *inc, "-c", os.path.join(CSRC, "fsdp_kernels.cu"),
         "-o", obj_k],
        [nvcc, *ARCH, *NVCC_FLAGS, *extra_nvcc, *inc, "-c", os.path.join(CSRC, "fsdp_noalloc.cu"),
         "-o", obj_n],
        [nvcc, *ARCH, *NVCC_FLAGS, *extra_nvcc, *inc, "-c", os.path.join(CSRC, "fsdp_bulk.cu"),
         "-o", obj_b],
        ["g++", *CXX_FLAGS, *inc, "-I", os.path.join(cuda, "include"), "-c",
         os.path.join(CSRC, "fsdp_capi.cpp"), "-o", obj_c],
    ]
    procs = [subprocess.Popen(j, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True) for j in jobs]
    failed = []
    for j, p in zip(jobs, procs):
        out, _ = p.communicate()
        if verbose or p.returncode:
            print(out, end="")
        if p.returncode:
            failed.append(" ".join(j))
    if failed:
        raise RuntimeError("compile failed: " + "; ".join(failed))
    tmp = os.path.join(LIB_DIR, f"{LIB_NAME}.{tag}")
    subprocess.run([nvcc, *ARCH, "-shared", "-cudart", "shared", obj_k, obj_n, obj_b, obj_c, "-o", tmp,
                    "-Xlinker", "-rpath," + os.path.join(cuda, "lib64")], check=True)
    os.replace(tmp, library_path())
    for o in (obj_k, obj_n, obj_b, obj_c):
        os.remove(o)
    return library_path()


if __name__ == "__main__":
    print(build(verbose=True))
