"""The allocation-free entry point (topk_transform_ragged_noalloc).

Some callers cannot allocate device memory at all: a plugin host may give a
library nothing but its input and output buffers, and a serving process may
reserve every byte of GPU memory up front for its KV cache. For them the
library offers one RAGGED entry point whose plan workspace is an array built
into the library. These tests call it through the C ABI and check that it
writes exactly what the ordinary plan + transform pair writes, on two calls
in a row (the built-in array keeps the previous call's contents, so the
second call must not depend on them). This file is collected last so that a
run stopping at the first failure has run every other test first.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_top_row_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DET = 1
CANARY = 0x7EADBEEF


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _reference(topk, w, flags):
    """The ordinary entry points, with a workspace torch allocates."""
    out = torch.full((w["batch"], w["k"]), CANARY, dtype=torch.int32, device="cuda")
    raw = torch.full_like(out, CANARY)
    topk.run_workload(w, out=out, out_raw=raw, flags=flags)
    return out, raw


def _noalloc(lib, w, flags):
    out = torch.full((w["batch"], w["k"]), CANARY, dtype=torch.int32, device="cuda")
    raw = torch.full_like(out, CANARY)
    st = lib.topk_transform_ragged_noalloc(
        _ptr(w["scores"]), int(w["score_stride"]), _ptr(w.get("row_starts")), _ptr(w["seq_lens"]),
        _ptr(w["out_offsets"]), int(w["batch"]), int(w["k"]), _ptr(out), _ptr(raw), flags,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, f"status {st}"
    return out, raw


@pytest.mark.parametrize("flags", [DET, 0])
def test_noalloc_matches_the_ordinary_entry_points_twice(cuda_lib, flags):
    lib = cuda_lib.load()
    cases = [
        wl.to_device(wl.mixed("cpu", mode="ragged", k=512, batch=40, max_len=70000, sub_id=7), "cuda"),
        wl.to_device(wl.ragged_tiny("cpu", sub_id=3), "cuda"),
    ]
    for w in cases:  # two calls in a row, on different inputs
        ref_out, ref_raw = _reference(cuda_lib, w, flags)
        out, raw = _noalloc(lib, w, flags)
        torch.cuda.synchronize()
        assert not bool((out == CANARY).any()) and not bool((raw == CANARY).any())
        if flags & DET:
            # the selected set is unique: sorted rows are bit-identical
            assert torch.equal(torch.sort(out, 1).values, torch.sort(ref_out, 1).values)
            assert torch.equal(torch.sort(raw, 1).values, torch.sort(ref_raw, 1).values)
        else:
            # equal scores may swap: the selected score bit patterns agree
            flat = w["scores"].reshape(-1).view(torch.int32)
            stride = int(w["score_stride"])
            starts = w["row_starts"].to(torch.int64)
            base = (torch.arange(w["batch"], device="cuda") * stride + starts)[:, None]
            def picked(r):
                idx = torch.where(r >= 0, base + r.to(torch.int64), torch.zeros_like(base))
                return torch.sort(torch.where(r >= 0, flat[idx], torch.full_like(r, -1)), 1).values
            assert torch.equal(picked(raw), picked(ref_raw))
            assert torch.equal((raw >= 0).sum(1), (ref_raw >= 0).sum(1))


def _det_equal(a, b):
    return torch.equal(torch.sort(a, 1).values, torch.sort(b, 1).values)


def test_noalloc_back_to_back_on_one_stream(cuda_lib):
    """Two calls queued on one stream with no synchronisation between them,
    on batches of different sizes and lengths (so the second call's plan
    rewrites the row lists the first call's kernels read): stream order alone
    keeps them apart, and each output matches the ordinary entry points."""
    lib = cuda_lib.load()
    a = wl.to_device(wl.mixed("cpu", mode="ragged", k=512, batch=40, max_len=70000, sub_id=11), "cuda")
    b = wl.to_device(wl.ragged_tiny("cpu", sub_id=4), "cuda")
    ref_a, _ = _reference(cuda_lib, a, DET)
    ref_b, _ = _reference(cuda_lib, b, DET)
    torch.cuda.synchronize()
    out_a, _ = _noalloc(lib, a, DET)
    out_b, _ = _noalloc(lib, b, DET)   # queued right behind the first call
    out_c, _ = _noalloc(lib, a, DET)   # and the first batch once more
    torch.cuda.synchronize()
    assert _det_equal(out_a, ref_a) and _det_equal(out_b, ref_b) and _det_equal(out_c, ref_a)


def test_noalloc_data_error_row_comes_out_empty(cuda_lib):
    """A row with a negative length is a data error: its slots all hold -1
    (this entry point does not report the error count), and the other rows
    are unaffected."""
    lib = cuda_lib.load()
    w = wl.mixed("cpu", mode="ragged", k=256, batch=6, max_len=40000, sub_id=13)
    w["seq_lens"] = w["seq_lens"].clone()
    w["seq_lens"][2] = -7
    d = wl.to_device(w, "cuda")
    ref_out, _ = _reference(cuda_lib, d, DET)
    out, raw = _noalloc(lib, d, DET)
    torch.cuda.synchronize()
    assert bool((out[2] == -1).all()) and bool((raw[2] == -1).all())
    assert _det_equal(out, ref_out)


def test_noalloc_rejects_a_batch_beyond_its_limit(cuda_lib):
    lib = cuda_lib.load()
    B = cuda_lib.TOPK_NOALLOC_MAX_BATCH + 1
    dummy = torch.zeros(4, dtype=torch.float32, device="cuda")
    ints = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    st = lib.topk_transform_ragged_noalloc(_ptr(dummy), 0, None, _ptr(ints), _ptr(ints), B, 16, _ptr(out), None,
                                           0, None)
    assert st == 5  # TOPK_ERR_WORKSPACE, nothing enqueued
