"""Build libzero_gb300.so (the C-ABI library with the sm_103a kernels) in-tree.

nvcc compiles each CUDA translation unit for sm_103a only and g++ the host
optimizer of the offload step, in parallel; nvcc then links one shared library
next to this file.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SOURCES = ["zero_kernels.cu", "zero_plan.cu", "zero_api.cu", "zero_group.cu", "zero_noalloc.cu"]
HOST_SOURCES = ["host_adam.cc"]
HEADERS = [os.path.join(CSRC, "zero_kernels.cuh"), os.path.join(CSRC, "zero_plan.h"),
           os.path.join(CSRC, "host_adam.h"),
           os.path.join(ROOT, "include", "zero.h"), os.path.join(ROOT, "include", "zero_debug.h")]
LIB = os.path.join(HERE, "libzero_gb300.so")
BUILD = os.path.join(HERE, "_build")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
CXX = os.environ.get("CXX", "g++")

# -fmad=false: no multiply-add contraction anywhere (the kernels also use
# explicit round-to-nearest intrinsics); no fast-math.
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
              "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", os.path.join(ROOT, "include"), "-I", CSRC]
# The host update: each fp32 operation rounded on its own (no contraction, no
# fast-math); -fno-math-errno only lets sqrt use the vector instruction.  No
# -march: the same flags build on x86-64 and aarch64.
CXX_FLAGS = ["-O3", "-std=c++17", "-fPIC", "-fvisibility=hidden", "-ffp-contract=off",
             "-fno-math-errno", "-pthread",
             "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    objs = []
    jobs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [path] + HEADERS):
            cmd = [NVCC, *NVCC_FLAGS, "-c", path, "-o", obj]
            if verbose_ptxas:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)
    for src in HOST_SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cc", ".o"))
        objs.append(obj)
        if force or _stale(obj, [path] + HEADERS):
            jobs.append([CXX, *CXX_FLAGS, "-c", path, "-o", obj])
    with ThreadPoolExecutor(max_workers=len(SOURCES) + len(HOST_SOURCES)) as ex:
        for r in ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs):
            if r.returncode != 0:
                raise RuntimeError("compile failed:\n" + r.stdout + r.stderr)
            if verbose_ptxas:
                sys.stderr.write(r.stderr)
    if force or _stale(LIB, objs):
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                        *objs, "-lpthread", "-o", tmp], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
