"""Compiles the C oracle (``pa_oracle.c``) into ``_build/liboracle.so``.

Test infrastructure: the product never links this library.
"""
from __future__ import annotations

import os
import subprocess
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
LIB = os.path.join(HERE, "_build", "liboracle.so")
CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False, src: str = SRC, out: Optional[str] = None) -> str:
    out = out or LIB
    if not force and out == LIB and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True))
