"""Builds the CUDA library in-tree (``_build/libtopk.so``) for sm_103a.

Four translation units (the plan and C ABI, the selection kernels compiled
for 512 and for 256 threads per row, and the indexer-logits kernel), compiled in parallel to
objects and linked into one shared library; one ``-gencode``, shared cudart
(the same runtime PyTorch loads). nvcc cross-compiles without a GPU.
"""

from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SOURCES = [os.path.join(CSRC, f) for f in ("topk.cu", "topk_select512.cu", "topk_select256.cu", "topk_logits.cu")]
HEADERS = [os.path.join(CSRC, f) for f in ("topk_common.cuh", "topk_select.cuh")]
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
    return any(os.path.getmtime(f) > t for f in (*SOURCES, *HEADERS, HEADER, __file__))


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and not needs_build():
        return LIB
    from concurrent.futures import ThreadPoolExecutor

    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = nvcc_path()
    tag = f".tmp{os.getpid()}"
    common = [nvcc, ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{os.path.join(ROOT, 'include')}",
              f"-I{CSRC}", *extra_flags]
    objs = [os.path.join(BUILD_DIR, os.path.basename(src) + tag + ".o") for src in SOURCES]

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = common + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        list(ex.map(compile_one, zip(SOURCES, objs)))
    tmp = LIB + tag
    link = [nvcc, ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp]
    for d in cuda_lib_dirs(nvcc):
        link += ["-Xlinker", f"-rpath,{d}"]
    if verbose:
        print(" ".join(link), flush=True)
    subprocess.run(link, check=True)
    for obj in objs:
        os.remove(obj)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []))
