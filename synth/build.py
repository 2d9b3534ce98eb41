"""Compiles the seeded input generator: host part (gcc) and device part (nvcc, sm_103a)."""
import os
import platform
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "_lib", platform.machine(), "libsynth_host.so")
DEV_LIB = os.path.join(HERE, "_lib", platform.machine(), "libsynth_dev.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _stale(out, srcs):
    return not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(s) for s in srcs)


def build_host(force=False):
    src = [os.path.join(HERE, "synth_host.c"), os.path.join(HERE, "synth.h")]
    if force or _stale(HOST_LIB, src):
        os.makedirs(os.path.dirname(HOST_LIB), exist_ok=True)
        tmp = HOST_LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                        src[0], "-o", tmp], check=True)
        os.replace(tmp, HOST_LIB)
    return HOST_LIB


def build_device(force=False):
    src = [os.path.join(HERE, "synth_dev.cu")]
    if force or _stale(DEV_LIB, src):
        os.makedirs(os.path.dirname(DEV_LIB), exist_ok=True)
        tmp = DEV_LIB + f".tmp{os.getpid()}"
        subprocess.run(["nvcc", *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-fmad=false",
                        src[0], "-o", tmp, "-lcudart"], check=True)
        os.replace(tmp, DEV_LIB)
    return DEV_LIB


def build(force=False):
    return build_host(force), build_device(force)


if __name__ == "__main__":
    print(build(force=True))
