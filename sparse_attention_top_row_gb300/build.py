"""Builds the CUDA library in-tree (``_build/libtopk.so``) for sm_103a.

One translation unit, one ``-gencode``, shared cudart (the same runtime
PyTorch loads). nvcc cross-compiles without a GPU.
"""

from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc", "topk.cu")
HEADER = os.path.join(ROOT, "include", "topk.h")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libtopk.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def cuda_lib_dirs(nvcc: str):
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    dirs = [os.path.join(root, "lib64"), os.path.join(root, "targets", "sbsa-linux", "lib"),
            os.path.join(root, "targets", "x86_64-linux", "lib")]
    return [d for d in dirs if os.path.isdir(d)]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in (SRC, HEADER, __file__))


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and not needs_build():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = nvcc_path()
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-cudart", "shared", f"-I{os.path.join(ROOT, 'include')}", SRC, "-o", tmp]
    for d in cuda_lib_dirs(nvcc):
        cmd += ["-Xlinker", f"-rpath,{d}"]
    cmd += list(extra_flags)
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []))
