"""Compile the CPU oracle (plain C: the FP64 layer and the integer trellis
encoder) into oracle/liboracle_exl3.so.

Test infrastructure: the library is loaded only by the tests, the smoke check
and the benchmark's CPU-baseline leg. -ffp-contract=off keeps every FP64
operation a separately rounded IEEE operation on x86-64 and on aarch64 alike.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRCS = [os.path.join(HERE, "exl3_oracle.c"), os.path.join(HERE, "exl3_encoder_oracle.c")]
LIB = os.path.join(HERE, "liboracle_exl3.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and all(os.path.getmtime(LIB) >= os.path.getmtime(s) for s in SRCS):
        return LIB
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", LIB + ".tmp"] + SRCS + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
