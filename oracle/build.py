"""Build the C++ oracle ``oracle/cpp/libmh3_oracle.so`` with g++.

TEST INFRASTRUCTURE ONLY: the library is the CPU oracle the tests, the smoke
check and the bench's CPU legs compare against.  Flags: -O2, OpenMP over
tokens, and -ffp-contract=off so that no multiply and add are fused (GCC
contracts them by default on Arm), which keeps every FP32 rounding point the
source states.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cpp", "mh3_oracle.cpp")
LIB = os.path.join(HERE, "cpp", "libmh3_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
         "-shared"]


def build(force: bool = False) -> str:
    """Compile if the source is newer than the library; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(
            os.path.getmtime(SRC), os.path.getmtime(__file__)):
        return LIB
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = ["g++", *FLAGS, SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"g++ failed for the oracle:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
