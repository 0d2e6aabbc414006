"""Oracle for the indexer top-k + transform: test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The library under
``sparse_attention_top_row_gb300`` never does.

The arithmetic lives in ``topk_oracle.cpp`` (plain single-threaded C++17,
sorted windows). This module only compiles it with g++ and marshals numpy
arrays through ctypes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "topk_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}

RAGGED = 0
PAGED = 1


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or one planted-mistake variant) into ``_build/``."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-shared", "-fPIC", f"-DORACLE_MUTANT={mutant}", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _LOCK:
        if mutant not in _LIBS:
            lib = ctypes.CDLL(build(mutant))
            fn = lib.oracle_topk_transform_packed
            fn.restype = ctypes.c_int64
            fn.argtypes = [
                ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
            ]
            _LIBS[mutant] = lib
        return _LIBS[mutant]


def _ptr(a):
    return None if a is None else a.ctypes.data


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def topk_transform(mode, scores, score_stride, row_starts, seq_lens, k, *,
                   out_offsets=None, page_table=None, page_table_stride=0, page_size=1,
                   page_table_row_starts=None, row_to_batch=None, batch=None, mutant: int = 0):
    """Run the oracle on host arrays.

    ``scores`` is a flat (or any contiguous) float32 array; row ``b``'s window
    begins at element ``b*score_stride + row_starts[b]``. PAGED rows may carry
    the packed layout's ``page_table_row_starts`` and ``row_to_batch``.
    Returns ``(out, out_raw, n_error_rows)`` with ``out``/``out_raw`` int32
    ``[batch, k]``. Selected positions are listed in ascending order, then
    ``-1`` padding.
    """
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    seq_lens = _i32(seq_lens)
    row_starts = _i32(row_starts)
    out_offsets = _i32(out_offsets)
    page_table = _i32(page_table)
    page_table_row_starts = _i32(page_table_row_starts)
    row_to_batch = _i32(row_to_batch)
    if batch is None:
        batch = int(seq_lens.shape[0])
    if mode == RAGGED and out_offsets is None:
        raise ValueError("RAGGED mode needs out_offsets")
    if mode == PAGED and page_table is None:
        raise ValueError("PAGED mode needs page_table")
    out = np.empty((batch, k), dtype=np.int32)
    out_raw = np.empty((batch, k), dtype=np.int32)
    errors = _load(mutant).oracle_topk_transform_packed(
        int(mode), _ptr(scores), int(score_stride), _ptr(row_starts), _ptr(seq_lens),
        _ptr(out_offsets), _ptr(page_table), int(page_table_stride), int(page_size),
        _ptr(page_table_row_starts), _ptr(row_to_batch), int(batch), int(k), _ptr(out), _ptr(out_raw))
    return out, out_raw, int(errors)


def run_workload(w, rows=None, mutant: int = 0):
    """Run the oracle on a workload dict (see the package's ``workloads``
    module), optionally on a subset of rows. Arrays may be torch tensors on any
    device; they are copied to host numpy first."""
    def host(x):
        if x is None:
            return None
        if hasattr(x, "detach"):
            return x.detach().cpu().numpy()
        return np.asarray(x)

    seq_lens = host(w["seq_lens"])
    row_starts = host(w.get("row_starts"))
    out_offsets = host(w.get("out_offsets"))
    page_table = host(w.get("page_table"))
    if page_table is not None:
        page_table = page_table.reshape(-1)
    pt_row_starts = host(w.get("page_table_row_starts"))
    row_to_batch = host(w.get("row_to_batch"))
    scores = host(w["scores"]).reshape(-1)
    stride = int(w["score_stride"])
    k = int(w["k"])
    mode = PAGED if w["mode"] == "paged" else RAGGED
    if rows is None:
        return topk_transform(mode, scores, stride, row_starts, seq_lens, k,
                              out_offsets=out_offsets, page_table=page_table,
                              page_table_stride=int(w.get("page_table_stride", 0)),
                              page_size=int(w.get("page_size", 1)),
                              page_table_row_starts=pt_row_starts, row_to_batch=row_to_batch, mutant=mutant)
    rows = np.asarray(rows, dtype=np.int64)
    outs, raws, errs = [], [], 0
    for b in rows:
        b = int(b)
        base = b * stride
        t = b if row_to_batch is None else int(row_to_batch[b])  # the row's page-table row
        pts = int(w.get("page_table_stride", 0))
        o, r, e = topk_transform(
            mode, scores[base:], 0,
            None if row_starts is None else row_starts[b:b + 1], seq_lens[b:b + 1], k,
            out_offsets=None if out_offsets is None else out_offsets[b:b + 1],
            page_table=None if page_table is None else page_table[t * pts:(t + 1) * pts],
            page_table_stride=pts, page_size=int(w.get("page_size", 1)),
            page_table_row_starts=None if pt_row_starts is None else pt_row_starts[b:b + 1],
            mutant=mutant)
        outs.append(o)
        raws.append(r)
        errs += e
    return np.concatenate(outs), np.concatenate(raws), errs


def swa_combine(out, out_raw, positions, window_size: int, swa_offsets, width: int, mutant: int = 0):
    """The SWA combine of the transform's rows (see topk_oracle.cpp): out,
    out_raw [B, k] int32 (numpy), positions [B], swa_offsets [B] or None;
    returns [B, width] int32."""
    lib = _load(mutant)
    fn = lib.oracle_swa_combine
    fn.restype = None
    fn.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    out = _i32(out)
    out_raw = _i32(out_raw)
    B, k = out.shape
    assert out_raw.shape == (B, k) and width >= k + window_size and window_size >= 0
    pos = _i32(positions)
    offs = None if swa_offsets is None else _i32(swa_offsets)
    res = np.empty((B, width), dtype=np.int32)
    fn(B, k, _ptr(out), _ptr(out_raw), _ptr(pos), int(window_size), _ptr(offs), int(width), _ptr(res))
    return res


def e4m3_value(code: int) -> float:
    """The value of one FP8 E4M3 code (see topk_oracle.cpp)."""
    fn = _load().oracle_e4m3_value
    fn.restype = ctypes.c_double
    fn.argtypes = [ctypes.c_uint8]
    return float(fn(int(code)))


def indexer_logits(q, kv, kv_scale, weights, ks, ke, out, mutant: int = 0):
    """Indexer logits (see topk_oracle.cpp) on host arrays: q uint8 E4M3 codes
    [n_q, heads, dim], kv uint8 [n_kv, dim], kv_scale float32 [n_kv], weights
    float32 [n_q, heads], ks/ke int32 [n_q]; `out` is a float32 [n_q, stride]
    array updated in place (only each row's window columns) and returned."""
    lib = _load(mutant)
    fn = lib.oracle_indexer_logits
    fn.restype = None
    fn.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                           ctypes.c_void_p, ctypes.c_int64]
    q = np.ascontiguousarray(q, dtype=np.uint8)
    kv = np.ascontiguousarray(kv, dtype=np.uint8)
    n_q, heads, dim = q.shape
    assert kv.ndim == 2 and kv.shape[1] == dim
    kv_scale = np.ascontiguousarray(kv_scale, dtype=np.float32)
    weights = np.ascontiguousarray(weights, dtype=np.float32).reshape(n_q, heads)
    ks = _i32(ks)
    ke = _i32(ke)
    assert out.dtype == np.float32 and out.ndim == 2 and out.shape[0] == n_q and out.flags.c_contiguous
    fn(_ptr(q), _ptr(kv), _ptr(kv_scale), _ptr(weights), _ptr(ks), _ptr(ke), int(n_q), int(heads), int(dim),
       int(kv.shape[0]), _ptr(out), int(out.shape[1]))
    return out


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def run_workload_threads(w, rows=None, threads=None, mutant: int = 0):
    """``run_workload`` with the rows split into ``threads`` contiguous blocks,
    each run on its own thread through the unchanged single-threaded routine
    (the C call releases the GIL, so the blocks run in parallel on the host
    cores). Returns the same ``(out, out_raw, n_error_rows)`` as
    ``run_workload`` over ``rows`` (all rows when None), in row order."""
    if rows is None:
        rows = np.arange(int(w["batch"]))
    rows = np.asarray(rows, dtype=np.int64)
    threads = max(1, min(threads or host_cores(), rows.size))
    if threads == 1:
        return run_workload(w, rows=rows, mutant=mutant)
    blocks = [b for b in np.array_split(rows, threads) if b.size]
    with ThreadPoolExecutor(len(blocks)) as ex:
        parts = list(ex.map(lambda b: run_workload(w, rows=b, mutant=mutant), blocks))
    return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]),
            sum(p[2] for p in parts))
