"""Compile the CUDA library in-tree for sm_103a (nvcc only, no cmake).

The result is ``mixed_precision_dense_gb300/_build/libmpgemm.so``; the
``ptxas -v`` report (registers, spills, shared memory per kernel) is kept
beside it in ``ptxas.txt``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libmpgemm.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _sources():
    return ([os.path.join(HERE, "csrc", "mpgemm.cu")],
            glob.glob(os.path.join(HERE, "csrc", "*")) + [os.path.join(ROOT, "include", "mpgemm.h")])


def nvcc_path() -> str:
    found = shutil.which("nvcc")
    if found:
        return found
    fallback = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(fallback):
        return fallback
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libmpgemm")


def build(force: bool = False) -> str:
    """Build libmpgemm.so if it is missing or older than its sources; return its path."""
    units, deps = _sources()
    os.makedirs(BUILD_DIR, exist_ok=True)
    report = os.path.join(BUILD_DIR, "ptxas.txt")
    if not force and os.path.exists(LIB_PATH) and os.path.exists(report):
        lib_time = os.path.getmtime(LIB_PATH)
        if all(os.path.getmtime(d) <= lib_time for d in deps):
            return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-std=c++17", "-lineinfo", "-Xptxas", "-v",
           "-Xcompiler", "-fPIC", "-shared", "-I", os.path.join(ROOT, "include"),
           "-o", tmp, *units]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    with open(report, "w") as f:
        f.write(" ".join(cmd) + "\n" + proc.stdout + proc.stderr)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc failed ({proc.returncode}):\n{proc.stderr[-4000:]}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True))
