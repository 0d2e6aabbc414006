"""The library inside a chain of kernels on one stream, as a serving loop
runs it: an upstream producer of the scores, the library's plan and
transform, and a downstream consumer of its output; launched directly and as
a replayed CUDA graph. Every output is compared with the CPU oracle.

The "#26788 [JIT Kernel] DeepSeek-V4 DSA indexer" page's review notes flag
two programmatic dependent launch (PDL) hazards: a kernel that lets its
dependents start before it has written its output, and ordering races around
that trigger. Here the producer triggers its dependents before it writes the
scores (after a delay, so an early read would see the stale buffer), and the
consumer is launched with the PDL attribute right after the library's
kernels, which also trigger early: the results are only right if every
kernel waits on its grid dependency before touching memory.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_top_row_gb300 import workloads as wl
from topk_checks import HostWorkload, compare_with_oracle

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
DET = 1
DELAY_CYCLES = 2_000_000   # about a millisecond of producer delay before it writes


@pytest.fixture(scope="module")
def chain():
    """The test-only producer / consumer kernels, built for sm_103a."""
    src = os.path.join(HERE, "pdl_chain.cu")
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(out_dir, "libpdl_chain.so")
    if not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run(["nvcc", "-gencode=arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler",
                        "-fPIC", "-cudart", "shared", src, "-o", tmp], check=True)
        os.replace(tmp, lib)
    import sparse_attention_top_row_gb300  # noqa: F401  (the shared CUDA runtime is loaded first)
    h = ctypes.CDLL(lib)
    h.pdl_produce.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong,
                              ctypes.c_int, ctypes.c_void_p]
    h.pdl_consume.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p]
    return h


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _workload(mode):
    # rows on the register, streaming and cluster routes, one launch
    return wl.mixed("cpu", mode=mode, k=1024, batch=24, max_len=70000, sub_id=31 if mode == "paged" else 32)


def _enqueue_chain(topk, chain, d, real, out, raw, copy, trigger, flags=DET):
    n = real.numel()
    assert chain.pdl_produce(_p(real), _p(d["scores"]), n, DELAY_CYCLES, trigger, _stream()) == 0
    topk.run_workload(d, out=out, out_raw=raw, flags=flags)
    assert chain.pdl_consume(_p(out), _p(copy), out.numel(), _stream()) == 0


def _check(w, copy, raw):
    hw = HostWorkload(w)
    ref_out, ref_raw, _ = oracle.run_workload(w)
    compare_with_oracle(hw, copy.cpu().numpy(), raw.cpu().numpy(), ref_out, ref_raw, deterministic=True)


@pytest.mark.parametrize("trigger", [1, 0])
@pytest.mark.parametrize("mode", ["paged", "ragged"])
def test_producer_library_consumer_chain(cuda_lib, chain, mode, trigger):
    """An early-triggering (or a never-triggering) producer, the library, a
    PDL consumer: the consumer's copy of the output matches the oracle on the
    scores the producer wrote, not on the stale buffer."""
    w = _workload(mode)
    d = wl.to_device(w, "cuda")
    real = d["scores"].clone()
    d["scores"].copy_(-real)                       # stale contents: the reversed order
    B, k = int(w["batch"]), int(w["k"])
    out = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    raw = torch.full_like(out, -7)
    copy = torch.full_like(out, -9)
    _enqueue_chain(cuda_lib, chain, d, real, out, raw, copy, trigger)
    torch.cuda.synchronize()
    _check(w, copy, raw)


@pytest.mark.parametrize("mode", ["paged", "ragged"])
def test_chain_captured_in_a_graph(cuda_lib, chain, mode):
    """The same chain captured once in a CUDA graph and replayed after new
    inputs are copied into the captured buffers (other lengths, other
    scores, another page table): every replay matches the oracle on its own
    inputs."""
    w1 = _workload(mode)
    w2 = wl.mixed("cpu", mode=mode, k=1024, batch=24, max_len=70000, sub_id=33)
    assert all(w1[key].shape == w2[key].shape for key in w1 if isinstance(w1[key], torch.Tensor))
    d = wl.to_device(w1, "cuda")
    real = torch.empty_like(d["scores"])
    B, k = int(w1["batch"]), int(w1["k"])
    out = torch.empty((B, k), dtype=torch.int32, device="cuda")
    raw = torch.empty_like(out)
    copy = torch.empty_like(out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _enqueue_chain(cuda_lib, chain, d, real, out, raw, copy, 1)
    for w in (w2, w1, w2):
        for key, v in w.items():
            if isinstance(v, torch.Tensor) and key != "scores":
                d[key].copy_(v)
        real.copy_(w["scores"])
        d["scores"].copy_(-real)
        out.fill_(-7)
        raw.fill_(-7)
        copy.fill_(-9)
        g.replay()
        torch.cuda.synchronize()
        _check(w, copy, raw)
