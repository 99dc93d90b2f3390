"""Build the scalar CPU oracle (test infrastructure only).

Compiles ``attn_res_ref.c`` with the host C compiler into
``oracle/_build/libattn_res_ref.so``.  No fast-math, no FMA contraction: the
oracle's double arithmetic must be plain IEEE operations in source order.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_res_ref.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libattn_res_ref.so")


def compile_source(src: str, lib: str) -> str:
    """Compile one C source of the oracle into a shared object at ``lib``."""
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-pthread", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def build(force: bool = False) -> str:
    """Compile the oracle if the shared object is missing or stale; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    return compile_source(SRC, LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
