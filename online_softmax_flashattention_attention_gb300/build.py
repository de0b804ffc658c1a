"""Build step: the CUDA library (nvcc for sm_103a, in-tree, one translation unit) and the
CPU library of the same operation (gcc, portable C11 with pthreads)."""
from __future__ import annotations

import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libattn.so")
SOURCES = [os.path.join(CSRC, "attn_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "attn.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in DEPS if os.path.exists(p))


CPU_SOURCE = os.path.join(HERE, "cpu", "attn_cpu.c")
CPU_LIB = os.path.join(HERE, "libattn_cpu.so")
CPU_DEPS = [CPU_SOURCE, os.path.join(ROOT, "include", "attn_cpu.h"), os.path.join(ROOT, "include", "attn.h")]
CPU_FLAGS = ["-O3", "-std=c11", "-fPIC", "-shared", "-fopenmp-simd", "-pthread"]


def build_cpu_library(force: bool = False) -> str:
    """Compile cpu/attn_cpu.c into libattn_cpu.so beside this file; returns its path."""
    if not force and os.path.exists(CPU_LIB) and all(
            os.path.getmtime(p) <= os.path.getmtime(CPU_LIB) for p in CPU_DEPS if os.path.exists(p)):
        return CPU_LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
    os.close(fd)
    try:
        subprocess.run(["gcc"] + CPU_FLAGS + [CPU_SOURCE, "-o", tmp, "-lm"], check=True, cwd=HERE)
        os.replace(tmp, CPU_LIB)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return CPU_LIB


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/ into libattn.so beside this file; returns its path."""
    if not force and up_to_date():
        return LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
    os.close(fd)
    cmd = [nvcc()] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else []) + SOURCES + ["-o", tmp]
    try:
        subprocess.run(cmd, check=True, cwd=HERE)
        os.replace(tmp, LIB)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
    print(build_cpu_library(force=True))
