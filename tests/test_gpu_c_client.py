"""The C ABI from a plain C program: tests/c_client/qr_c_client.c, compiled
with gcc as C11 against include/qr.h and linked to libqr.so (and, for its
checks, the C oracle and the CUDA runtime), runs every code width through the
fused, unfused and two-shot entry points, and every codec through the
per-rank two-shot calls, and compares each wire and output with the oracle's;
see the program's header."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    pytest.skip("no CUDA toolkit headers")


def test_plain_c_program(tmp_path):
    from bit_quantized_all_gb300 import build
    lib = build.build()
    import oracle
    orc = oracle.build()
    cuda = _cuda_home()
    exe = tmp_path / "qr_c_client"
    libdir = os.path.dirname(lib)
    orcdir = os.path.dirname(orc)
    cudalib = os.path.join(cuda, "lib64")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "oracle"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_client", "qr_c_client.c"), "-o", str(exe),
           lib, orc, "-L", cudalib, "-lcudart",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{orcdir}", f"-Wl,-rpath,{cudalib}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    p = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stdout + p.stderr
    assert "qr_c_client ok" in p.stdout
