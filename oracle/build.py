"""Build the CPU oracle (test infrastructure) into oracle/_build/libmoe_oracle.so.

Plain gcc, no fused multiply-add contraction (the oracle calls fmaf where the
combine definition fuses), no fast-math. Builds the same on x86_64 and aarch64.
"""
from __future__ import annotations

import os
import subprocess
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libmoe_oracle.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    # unique per process and thread: concurrent first builds never share a file
    tmp = LIB + f".tmp{os.getpid()}.{threading.get_ident()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-Wall",
           "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
