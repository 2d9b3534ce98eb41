"""Compiles the oracle (C, OpenMP) into oracle/_lib/liboracle.so. Test infrastructure."""
import os
import platform
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "_lib", platform.machine(), "liboracle.so")
SOURCES = [os.path.join(HERE, "oracle.c"), os.path.join(HERE, "source.c"),
           os.path.join(HERE, "..", "synth", "synth_host.c")]


def build(force: bool = False) -> str:
    newest = max(os.path.getmtime(p) for p in SOURCES + [os.path.join(HERE, "oracle.h")])
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-Wall", "-Wno-unused-function", *SOURCES, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
