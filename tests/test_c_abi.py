"""The C ABI from plain C: the header compiles as strict C11 on its own, and
a C program (tests/c/abi_check.c) drives plan queries, the unshard, the
fused gradient sync and apply through it with cudaMalloc'd buffers, no
Python in between, checking closed-form results."""
import glob
import os
import shutil
import subprocess

import pytest

from hsdp_sharded_parameter_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
DRIVER = os.path.join(ROOT, "tests", "c", "abi_check.c")
C11 = ["-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic"]


def _gcc():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    return gcc


def _cuda_dirs():
    try:
        home = B.cuda_home()
    except RuntimeError:
        pytest.skip("CUDA toolkit not found")
    inc = os.path.join(home, "include")
    libs = [d for d in [os.path.join(home, "lib64")] + glob.glob(os.path.join(home, "targets", "*", "lib"))
            if os.path.exists(os.path.join(d, "libcudart.so"))]
    return inc, libs


def test_header_is_self_contained_c11(tmp_path):
    src = tmp_path / "only_header.c"
    src.write_text('#include "hsdp_fsdp.h"\nint main(void) { return FSDP_OK; }\n')
    subprocess.run([_gcc(), *C11, "-I", INCLUDE, "-fsyntax-only", str(src)], check=True)


def test_c_driver_compiles_as_c11():
    inc, _ = _cuda_dirs()
    subprocess.run([_gcc(), *C11, "-I", INCLUDE, "-I", inc, "-fsyntax-only", DRIVER], check=True)


@pytest.mark.gpu
def test_c_driver_runs(tmp_path):
    inc, libs = _cuda_dirs()
    if not libs:
        pytest.skip("libcudart.so not found")
    lib = B.library_path()
    assert os.path.exists(lib), "build the library first"
    exe = tmp_path / "abi_check"
    libdir = os.path.dirname(lib)
    rpath = ":".join([libdir, *libs])
    subprocess.run([_gcc(), *C11, "-O1", "-I", INCLUDE, "-I", inc, DRIVER, "-o", str(exe),
                    "-L", libdir, "-lhsdp_fsdp", *[f"-L{d}" for d in libs], "-lcudart",
                    f"-Wl,-rpath,{rpath}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_check: ok" in r.stdout
