"""Build the C oracle (``oracle/ref_attn.c``) into ``oracle/liboracle_attn.so``.

Test infrastructure only. Plain gcc, portable flags (the same source builds on
x86-64 and aarch64 hosts): no ``-march=native``, no intrinsics.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ref_attn.c")
LIB = os.path.join(HERE, "liboracle_attn.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
