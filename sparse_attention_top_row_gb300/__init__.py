"""Sparse-attention indexer top-k + transform on GB300: Python binding.

Thin ctypes marshalling over the C ABI of ``include/topk.h`` (the
``_build/libtopk.so`` library): the functions take torch CUDA tensors, check
each one's dtype, device, size and layout, pass their device pointers and the
current CUDA stream, and raise on a non-zero status. Every step of the computation runs in the library's CUDA kernels;
there is no fallback of any kind, and calling without the built library
raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import workloads  # noqa: F401  (seeded synthetic inputs)

TOPK_MAX_K = 2048
TOPK_DETERMINISTIC = 1
TOPK_DEVICE_FLAG_PLAN_MISMATCH = 1
TOPK_DEVICE_FLAG_INTERNAL = 2
TOPK_DEVICE_FLAG_TIMEOUT = 4

STATUS = {0: "TOPK_OK", 1: "TOPK_ERR_ARG", 2: "TOPK_ERR_ALIGN", 3: "TOPK_ERR_K",
          4: "TOPK_ERR_PAGE_SIZE", 5: "TOPK_ERR_WORKSPACE", 6: "TOPK_ERR_CUDA"}

_LIB = None
_LOCK = threading.Lock()
_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtopk.so")

EXPORTED = ("topk_workspace_bytes", "topk_plan", "topk_transform_paged", "topk_transform_paged_packed",
            "topk_transform_ragged", "topk_read_device_errors", "topk_status_string",
            "topk_transform_ragged_noalloc", "topk_transform_launches", "topk_transform_ragged_swa",
            "topk_indexer_logits")
TOPK_INDEXER_HEADS = 64
TOPK_INDEXER_DIM = 128
TOPK_NOALLOC_MAX_BATCH = 16384


class TopKError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads the built library (``build()`` in ``__graft_entry__`` or
    ``python -m sparse_attention_top_row_gb300.build`` makes it)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing")
        import torch  # noqa: F401  (loads the shared CUDA runtime first)
        lib = ctypes.CDLL(path)
        c_i32, c_i64, c_u32, c_sz, c_p = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                          ctypes.c_size_t, ctypes.c_void_p)
        lib.topk_workspace_bytes.restype = c_sz
        lib.topk_workspace_bytes.argtypes = [c_i32]
        lib.topk_plan.restype = ctypes.c_int
        lib.topk_plan.argtypes = [c_p, c_i32, c_i32, c_p, c_sz, c_p]
        lib.topk_transform_paged.restype = ctypes.c_int
        lib.topk_transform_paged.argtypes = [c_p, c_i64, c_p, c_p, c_p, c_i64, c_i32, c_i32, c_i32,
                                             c_p, c_sz, c_p, c_p, c_u32, c_p]
        lib.topk_transform_paged_packed.restype = ctypes.c_int
        lib.topk_transform_paged_packed.argtypes = [c_p, c_i64, c_p, c_p, c_p, c_i64, c_i32, c_p, c_p, c_i32, c_i32,
                                                    c_p, c_sz, c_p, c_p, c_u32, c_p]
        lib.topk_transform_ragged.restype = ctypes.c_int
        lib.topk_transform_ragged.argtypes = [c_p, c_i64, c_p, c_p, c_p, c_i32, c_i32,
                                              c_p, c_sz, c_p, c_p, c_u32, c_p]
        lib.topk_read_device_errors.restype = ctypes.c_int
        lib.topk_read_device_errors.argtypes = [c_p, ctypes.POINTER(c_i32), ctypes.POINTER(c_u32), c_p]
        lib.topk_transform_ragged_noalloc.restype = ctypes.c_int
        lib.topk_transform_ragged_noalloc.argtypes = [c_p, c_i64, c_p, c_p, c_p, c_i32, c_i32, c_p, c_p, c_u32, c_p]
        lib.topk_transform_ragged_swa.restype = ctypes.c_int
        lib.topk_transform_ragged_swa.argtypes = [c_p, c_i64, c_p, c_p, c_p, c_i32, c_i32, c_p, c_sz,
                                                  c_p, c_i32, c_p, c_i32, c_p, c_p, c_u32, c_p]
        lib.topk_indexer_logits.restype = ctypes.c_int
        lib.topk_indexer_logits.argtypes = [c_p, c_p, c_p, c_p, c_p, c_p, c_i32, c_i32, c_p, c_i64, c_p, c_p]
        lib.topk_transform_launches.restype = ctypes.c_int
        lib.topk_transform_launches.argtypes = [c_i32]
        lib.topk_status_string.restype = ctypes.c_char_p
        lib.topk_status_string.argtypes = [ctypes.c_int]
        _LIB = lib
        return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _arg(t, name, dtype=None, numel=0, required=True, dense=True, device=None):
    """Checks one tensor argument before its pointer crosses the C ABI: a CUDA
    tensor on `device` (the index of the device the call launches on) of the
    given dtype, at least `numel` elements, dense (row arrays, outputs, the
    workspace) or with a unit innermost stride (arrays whose row stride is a
    separate argument). None passes where the argument is optional (or the
    batch is empty). Raises TypeError / ValueError; returns the pointer.
    The common case costs a handful of attribute reads."""
    if t is None:
        if required and numel > 0:
            raise ValueError(f"{name} is required")
        return None
    try:
        ok = ((dtype is None or t.dtype is dtype) and t.is_cuda
              and (device is None or t.get_device() == device)
              and (t.is_contiguous() if dense else (t.dim() == 0 or t.numel() <= 1 or t.stride(-1) == 1))
              and t.numel() >= numel)
    except AttributeError:
        ok = False
    if not ok:
        _reject(t, name, dtype, numel, dense, device)
    return ctypes.c_void_p(t.data_ptr())


def _reject(t, name, dtype, numel, dense, device=None):
    """Raises the error that says why `t` failed `_arg`."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (it is on {t.device})")
    if device is not None and t.get_device() != device:
        raise ValueError(f"{name} is on cuda:{t.get_device()}, but the call runs on cuda:{device}")
    if dense and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not dense and t.dim() > 0 and t.numel() > 1 and t.stride(-1) != 1:
        raise ValueError(f"{name} must have a unit innermost stride")
    raise ValueError(f"{name} has {t.numel()} elements, fewer than the {numel} required")


def _strided_numel(batch, stride):
    """Fewest elements a buffer of `batch` rows `stride` apart can hold: the
    last row starts at (batch - 1) * stride and holds at least one element."""
    return 0 if batch == 0 else (batch - 1) * max(int(stride), 0) + 1


def _rows(seq_lens, device):
    """The batch, from seq_lens (a CUDA int32 vector, one entry per row)."""
    import torch
    if seq_lens is None:
        raise ValueError("seq_lens is required")
    _arg(seq_lens, "seq_lens", torch.int32, device=device)
    return int(seq_lens.numel())


def _ws(workspace, device=None):
    """The workspace pointer and its size in bytes (any dtype; dense)."""
    if workspace is None:
        raise ValueError("workspace is required")
    return _arg(workspace, "workspace", device=device), workspace.numel() * workspace.element_size()


def _stream(stream):
    """The stream handle and the index of the device the call launches on
    (the current device; a given stream must belong to it). Without CUDA
    there is no device: the tensor checks then reject every argument (none can
    be a CUDA tensor) before anything else happens."""
    import torch
    if not torch.cuda.is_available():
        return None, None
    dev = torch.cuda.current_device()
    s = stream if stream is not None else torch.cuda.current_stream()
    if s.device.index is not None and s.device.index != dev:
        raise ValueError(f"the stream belongs to cuda:{s.device.index}, but cuda:{dev} is current")
    return ctypes.c_void_p(s.cuda_stream), dev


def _check(fn, status):
    if status != 0:
        raise TopKError(fn, status)


def topk_workspace_bytes(batch: int) -> int:
    return int(load().topk_workspace_bytes(int(batch)))


def topk_transform_launches(batch: int) -> int:
    """Kernels one transform of `batch` rows launches on the current device
    (1 or 2; 0 for an empty batch)."""
    n = int(load().topk_transform_launches(int(batch)))
    if n < 0:
        raise TopKError("topk_transform_launches", 6)
    return n


def new_workspace(batch: int, device="cuda"):
    """A workspace tensor of topk_workspace_bytes(batch) bytes (torch owns it)."""
    import torch
    return torch.empty(topk_workspace_bytes(batch), dtype=torch.uint8, device=device)


def topk_plan(seq_lens, k: int, workspace, stream=None):
    lib = load()
    st, dev = _stream(stream)
    batch = _rows(seq_lens, dev)
    ws, ws_bytes = _ws(workspace, dev)
    _check("topk_plan", lib.topk_plan(_ptr(seq_lens), batch, int(k), ws, ws_bytes, st))


def topk_transform_paged(scores, score_stride: int, row_starts, seq_lens, page_table,
                         page_table_stride: int, page_size: int, k: int, workspace, out,
                         out_raw=None, flags: int = 0, stream=None):
    import torch
    lib = load()
    st, dev = _stream(stream)
    batch = _rows(seq_lens, dev)
    i32 = torch.int32
    args = (_arg(scores, "scores", torch.float32, _strided_numel(batch, score_stride), dense=False, device=dev),
            int(score_stride), _arg(row_starts, "row_starts", i32, batch, required=False, device=dev),
            _ptr(seq_lens),
            _arg(page_table, "page_table", i32, _strided_numel(batch, page_table_stride), dense=False, device=dev),
            int(page_table_stride), int(page_size), batch, int(k), *_ws(workspace, dev),
            _arg(out, "out", i32, batch * int(k), device=dev),
            _arg(out_raw, "out_raw", i32, batch * int(k), required=False, device=dev), int(flags))
    _check("topk_transform_paged", lib.topk_transform_paged(*args, st))


def topk_transform_paged_packed(scores, score_stride: int, row_starts, seq_lens, page_table,
                                page_table_stride: int, page_size: int, page_table_row_starts, row_to_batch,
                                k: int, workspace, out, out_raw=None, flags: int = 0, stream=None):
    import torch
    lib = load()
    st, dev = _stream(stream)
    batch = _rows(seq_lens, dev)
    i32 = torch.int32
    # with row_to_batch the table's row count is the caller's; without it,
    # row b reads table row b
    pt_rows = (1 if batch else 0) if row_to_batch is not None else batch
    args = (_arg(scores, "scores", torch.float32, _strided_numel(batch, score_stride), dense=False, device=dev),
            int(score_stride), _arg(row_starts, "row_starts", i32, batch, required=False, device=dev),
            _ptr(seq_lens),
            _arg(page_table, "page_table", i32, _strided_numel(pt_rows, page_table_stride), dense=False,
                 device=dev),
            int(page_table_stride), int(page_size),
            _arg(page_table_row_starts, "page_table_row_starts", i32, batch, required=False, device=dev),
            _arg(row_to_batch, "row_to_batch", i32, batch, required=False, device=dev), batch, int(k),
            *_ws(workspace, dev), _arg(out, "out", i32, batch * int(k), device=dev),
            _arg(out_raw, "out_raw", i32, batch * int(k), required=False, device=dev), int(flags))
    _check("topk_transform_paged_packed", lib.topk_transform_paged_packed(*args, st))


def topk_transform_ragged(scores, score_stride: int, row_starts, seq_lens, out_offsets, k: int,
                          workspace, out, out_raw=None, flags: int = 0, stream=None):
    import torch
    lib = load()
    st, dev = _stream(stream)
    batch = _rows(seq_lens, dev)
    i32 = torch.int32
    args = (_arg(scores, "scores", torch.float32, _strided_numel(batch, score_stride), dense=False, device=dev),
            int(score_stride), _arg(row_starts, "row_starts", i32, batch, required=False, device=dev),
            _ptr(seq_lens), _arg(out_offsets, "out_offsets", i32, batch, device=dev), batch, int(k),
            *_ws(workspace, dev), _arg(out, "out", i32, batch * int(k), device=dev),
            _arg(out_raw, "out_raw", i32, batch * int(k), required=False, device=dev), int(flags))
    _check("topk_transform_ragged", lib.topk_transform_ragged(*args, st))


def topk_transform_ragged_swa(scores, score_stride: int, row_starts, seq_lens, out_offsets, k: int, workspace,
                              positions, window_size: int, swa_offsets, out_width: int, out, out_raw=None,
                              flags: int = 0, stream=None):
    """RAGGED top-k fused with the SWA combine: out is [batch, out_width]
    (see include/topk.h)."""
    import torch
    lib = load()
    st, dev = _stream(stream)
    batch = _rows(seq_lens, dev)
    i32 = torch.int32
    args = (_arg(scores, "scores", torch.float32, _strided_numel(batch, score_stride), dense=False, device=dev),
            int(score_stride), _arg(row_starts, "row_starts", i32, batch, required=False, device=dev),
            _ptr(seq_lens), _arg(out_offsets, "out_offsets", i32, batch, device=dev), batch, int(k),
            *_ws(workspace, dev), _arg(positions, "positions", i32, batch, device=dev), int(window_size),
            _arg(swa_offsets, "swa_offsets", i32, batch, required=False, device=dev), int(out_width),
            _arg(out, "out", i32, batch * int(out_width), device=dev),
            _arg(out_raw, "out_raw", i32, batch * int(k), required=False, device=dev), int(flags))
    _check("topk_transform_ragged_swa", lib.topk_transform_ragged_swa(*args, st))


def topk_transform_ragged_noalloc(scores, score_stride: int, row_starts, seq_lens, out_offsets, k: int, out,
                                  out_raw=None, flags: int = 0, stream=None):
    """Plan + RAGGED transform without a caller workspace (the library's
    built-in one; batch <= TOPK_NOALLOC_MAX_BATCH). See include/topk.h."""
    import torch
    lib = load()
    st, dev = _stream(stream)
    batch = _rows(seq_lens, dev)
    i32 = torch.int32
    args = (_arg(scores, "scores", torch.float32, _strided_numel(batch, score_stride), dense=False, device=dev),
            int(score_stride), _arg(row_starts, "row_starts", i32, batch, required=False, device=dev),
            _ptr(seq_lens), _arg(out_offsets, "out_offsets", i32, batch, device=dev), batch, int(k),
            _arg(out, "out", i32, batch * int(k), device=dev),
            _arg(out_raw, "out_raw", i32, batch * int(k), required=False, device=dev), int(flags))
    _check("topk_transform_ragged_noalloc", lib.topk_transform_ragged_noalloc(*args, st))


def topk_indexer_logits(q, kv, kv_scale, weights, ks, ke, logits, logits_stride: int, device_flags, stream=None):
    """Indexer logits (see include/topk.h): q [n_q, 64, 128] and kv [n_kv, 128]
    FP8 E4M3 codes (torch.uint8 or torch.float8_e4m3fn), kv_scale float32
    [n_kv], weights float32 [n_q, 64], ks/ke int32 [n_q]; row t of `logits`
    (float32, rows logits_stride apart) gets columns ks[t] .. ke[t] - 1;
    device_flags: an int32 word the kernel ORs TOPK_DEVICE_FLAG_TIMEOUT into."""
    import torch
    lib = load()
    st, dev = _stream(stream)
    for name, t, nd in (("q", q, 3), ("kv", kv, 2)):
        if not isinstance(t, torch.Tensor) or t.dim() != nd or t.shape[-1] != TOPK_INDEXER_DIM or \
                (nd == 3 and t.shape[1] != TOPK_INDEXER_HEADS):
            raise ValueError(f"{name} must be a tensor of shape {'[n_q, 64, 128]' if nd == 3 else '[n_kv, 128]'}")
    if q.dtype is torch.float8_e4m3fn:
        q = q.view(torch.uint8)
    if kv.dtype is torch.float8_e4m3fn:
        kv = kv.view(torch.uint8)
    n_q, n_kv = int(q.shape[0]), int(kv.shape[0])
    u8, f32, i32 = torch.uint8, torch.float32, torch.int32
    need = 0 if n_q == 0 or n_kv == 0 else (n_q - 1) * max(int(logits_stride), 0) + n_kv
    args = (_arg(q, "q", u8, n_q * TOPK_INDEXER_HEADS * TOPK_INDEXER_DIM, device=dev),
            _arg(kv, "kv", u8, n_kv * TOPK_INDEXER_DIM, device=dev),
            _arg(kv_scale, "kv_scale", f32, n_kv, device=dev),
            _arg(weights, "weights", f32, n_q * TOPK_INDEXER_HEADS, device=dev),
            _arg(ks, "ks", i32, n_q, device=dev), _arg(ke, "ke", i32, n_q, device=dev), n_q, n_kv,
            _arg(logits, "logits", f32, need, dense=False, device=dev), int(logits_stride),
            _arg(device_flags, "device_flags", i32, 1, device=dev))
    _check("topk_indexer_logits", lib.topk_indexer_logits(*args, st))


def topk_read_device_errors(workspace, stream=None):
    """Returns (error_rows, flags); synchronises the stream."""
    lib = load()
    n = ctypes.c_int32(0)
    f = ctypes.c_uint32(0)
    st, dev = _stream(stream)
    ws, _ = _ws(workspace, dev)
    _check("topk_read_device_errors", lib.topk_read_device_errors(ws, ctypes.byref(n), ctypes.byref(f), st))
    return int(n.value), int(f.value)


def run_workload(w, out=None, out_raw=None, workspace=None, flags: int = 0, plan: bool = True,
                 stream=None):
    """Plan + transform on a workload dict whose tensors are on the GPU.
    Returns (out, out_raw, workspace)."""
    import torch
    dev = w["scores"].device
    B, k = int(w["batch"]), int(w["k"])
    swa = w.get("positions") is not None
    if out is None:
        out = torch.empty((B, int(w["out_width"]) if swa else k), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = new_workspace(B, dev)
    if plan:
        topk_plan(w["seq_lens"], k, workspace, stream=stream)
    if w["mode"] == "paged" and (w.get("page_table_row_starts") is not None or w.get("row_to_batch") is not None):
        topk_transform_paged_packed(w["scores"], w["score_stride"], w.get("row_starts"), w["seq_lens"],
                                    w["page_table"], w["page_table_stride"], w["page_size"],
                                    w.get("page_table_row_starts"), w.get("row_to_batch"), k, workspace,
                                    out, out_raw, flags, stream=stream)
    elif w["mode"] == "paged":
        topk_transform_paged(w["scores"], w["score_stride"], w.get("row_starts"), w["seq_lens"],
                             w["page_table"], w["page_table_stride"], w["page_size"], k, workspace,
                             out, out_raw, flags, stream=stream)
    elif swa:
        topk_transform_ragged_swa(w["scores"], w["score_stride"], w.get("row_starts"), w["seq_lens"],
                                  w["out_offsets"], k, workspace, w["positions"], w["window_size"],
                                  w.get("swa_offsets"), w["out_width"], out, out_raw, flags, stream=stream)
    else:
        topk_transform_ragged(w["scores"], w["score_stride"], w.get("row_starts"), w["seq_lens"],
                              w["out_offsets"], k, workspace, out, out_raw, flags, stream=stream)
    return out, out_raw, workspace
