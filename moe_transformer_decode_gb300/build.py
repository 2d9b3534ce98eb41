"""Builds libmk.so (the decode library, CUDA for sm_103a) in-tree under _lib/."""
import os
import platform
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_lib", platform.machine())
LIB = os.path.join(OUT, "libmk.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
UNITS = ["mk_kernel.cu", "mk_host.cpp", "mk_static.cu"]
HEADERS = [os.path.join(CSRC, "mk_internal.h"), os.path.join(ROOT, "include", "mk.h")]


def _stale(out, deps):
    return not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(d) for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    objs = []
    jobs = []
    for u in UNITS:
        src = os.path.join(CSRC, u)
        obj = os.path.join(OUT, u + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + HEADERS):
            cmd = ["nvcc", *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-c", src, "-o", obj,
                   "-I", os.path.join(ROOT, "include")]
            if u.endswith(".cu"):
                cmd += ["-Xptxas", "-v"] if verbose else []
            else:
                cmd[cmd.index("-c"):cmd.index("-c")] = ["-x", "cu"]
            jobs.append(cmd)
    with ThreadPoolExecutor(max_workers=len(jobs) or 1) as ex:
        for r in ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs):
            if r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
                raise RuntimeError("nvcc failed")
            if verbose:
                sys.stderr.write(r.stdout + r.stderr)
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["nvcc", *ARCH, "-shared", *objs, "-o", tmp, "-lcudart"], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
