"""The C ABI from a plain C program (tests/c_abi_ce.c): built with gcc against
include/vlmce.h and lib/libvlmce.so, run on the GPU, checked against the
closed form inside the program."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_caller(tmp_path):
    from vocabulary_lm_cross_gb300 import build
    lib = build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cc = shutil.which("gcc") or shutil.which("cc")
    assert cc, "a C compiler is required"
    exe = str(tmp_path / "c_abi_ce")
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-O2", "-std=c11", os.path.join(ROOT, "tests", "c_abi_ce.c"), "-o", exe,
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    "-L", libdir, f"-Wl,-rpath,{libdir}", "-lvlmce",
                    "-L", os.path.join(cuda, "lib64"), f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}",
                    "-lcudart", "-lm"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
