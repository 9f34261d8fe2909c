"""Compile the CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain g++, C++17, -O2 without fast-math and with -ffp-contract=off, so every
floating-point operation is the IEEE operation the source names.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dllm_oracle.cpp")
HDR = os.path.join(HERE, "dllm_oracle.h")
LIB = os.path.join(HERE, "liboracle.so")


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR, __file__))


def build(force: bool = False) -> str:
    if force or needs_build():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
               "-o", tmp, SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
