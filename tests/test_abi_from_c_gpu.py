"""The C ABI from a plain C program (tests/abi_from_c.c): built with the host
C compiler against include/attn_res.h, linked with libattn_res.so, the CUDA
runtime and the oracle's shared library, and run once; it checks one call on
padded rows against the oracle and the argument errors, and prints "ok"."""
import os
import subprocess

import pytest

from attention_residual_fusion_gb300 import _build
from oracle import build as oracle_build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_abi_from_plain_c(tmp_path):
    lib = _build.build()
    ref = oracle_build.build()
    exe = str(tmp_path / "abi_from_c")
    libdirs = [os.path.dirname(lib), os.path.dirname(ref), os.path.join(CUDA, "lib64")]
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-o", exe,
           os.path.join(ROOT, "tests", "abi_from_c.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include")]
    for d in libdirs:
        cmd += ["-L", d, f"-Wl,-rpath,{d}"]
    cmd += ["-lattn_res", "-lattn_res_ref", "-lcudart", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
