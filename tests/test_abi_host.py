"""The C-ABI library loads and exports every declared symbol; host-side
argument checks return their documented status codes. No GPU work: every call
below fails validation before anything is enqueued."""

from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "topk.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_top_row_gb300 import build as b
    b.build()
    import sparse_attention_top_row_gb300 as topk
    return topk.load()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"TOPK_API\s+[\w\s\*]+?\b(topk_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    assert {"topk_plan", "topk_transform_paged", "topk_transform_ragged",
            "topk_workspace_bytes", "topk_read_device_errors"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_transform_launches_of_an_empty_batch(lib):
    assert lib.topk_transform_launches(0) == 0 and lib.topk_transform_launches(-3) == 0


def test_workspace_bytes(lib):
    assert lib.topk_workspace_bytes(-1) == 0
    assert lib.topk_workspace_bytes(0) == 256
    assert lib.topk_workspace_bytes(48) == 512          # 64 + 2*4*48 = 448 -> 512
    assert lib.topk_workspace_bytes(16384) % 256 == 0
    assert lib.topk_workspace_bytes(16384) >= 64 + 8 * 16384


FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: validation fails first
FAKE_UNALIGNED = ctypes.c_void_p(0x10004)


def test_plan_validation(lib):
    ws = lib.topk_workspace_bytes(8)
    assert lib.topk_plan(FAKE, 8, 0, FAKE, ws, None) == 3
    assert lib.topk_plan(FAKE, 8, 2049, FAKE, ws, None) == 3
    assert lib.topk_plan(FAKE, -1, 16, FAKE, ws, None) == 1
    assert lib.topk_plan(None, 8, 16, FAKE, ws, None) == 1
    assert lib.topk_plan(FAKE, 8, 16, None, ws, None) == 5
    assert lib.topk_plan(FAKE, 8, 16, FAKE, ws - 1, None) == 5


def test_transform_validation(lib):
    ws = lib.topk_workspace_bytes(8)
    paged = lib.topk_transform_paged
    ragged = lib.topk_transform_ragged
    # scores, stride, row_starts, seq_lens, page_table, pt_stride, page_size, batch, k, ws, ws_bytes, out, out_raw, flags, stream
    assert paged(FAKE, 64, None, FAKE, FAKE, 4, 64, 8, 0, FAKE, ws, FAKE, None, 0, None) == 3
    assert paged(FAKE, 62, None, FAKE, FAKE, 4, 64, 8, 16, FAKE, ws, FAKE, None, 0, None) == 1
    assert paged(FAKE, -4, None, FAKE, FAKE, 4, 64, 8, 16, FAKE, ws, FAKE, None, 0, None) == 1
    assert paged(FAKE_UNALIGNED, 64, None, FAKE, FAKE, 4, 64, 8, 16, FAKE, ws, FAKE, None, 0, None) == 2
    assert paged(FAKE, 64, None, FAKE, FAKE, 4, 48, 8, 16, FAKE, ws, FAKE, None, 0, None) == 4
    assert paged(FAKE, 64, None, FAKE, FAKE, 4, 0, 8, 16, FAKE, ws, FAKE, None, 0, None) == 4
    assert paged(FAKE, 64, None, FAKE, FAKE, 4, 1 << 20, 8, 16, FAKE, ws, FAKE, None, 0, None) == 4
    assert paged(FAKE, 64, None, FAKE, None, 4, 64, 8, 16, FAKE, ws, FAKE, None, 0, None) == 1
    assert paged(FAKE, 64, None, FAKE, FAKE, -1, 64, 8, 16, FAKE, ws, FAKE, None, 0, None) == 1
    assert paged(FAKE, 64, None, None, FAKE, 4, 64, 8, 16, FAKE, ws, FAKE, None, 0, None) == 1
    assert paged(FAKE, 64, None, FAKE, FAKE, 4, 64, 8, 16, FAKE, ws, None, None, 0, None) == 1
    assert paged(FAKE, 64, None, FAKE, FAKE, 4, 64, 8, 16, FAKE, ws - 1, FAKE, None, 0, None) == 5
    assert paged(FAKE, 64, None, FAKE, FAKE, 4, 64, -2, 16, FAKE, ws, FAKE, None, 0, None) == 1
    # flags: TOPK_DETERMINISTIC is the only bit
    assert paged(FAKE, 64, None, FAKE, FAKE, 4, 64, 8, 16, FAKE, ws, FAKE, None, 2, None) == 1
    assert paged(FAKE, 64, None, FAKE, FAKE, 4, 64, 8, 16, FAKE, ws, FAKE, None, 1 << 31, None) == 1
    # scores, stride, row_starts, seq_lens, out_offsets, batch, k, ws, ws_bytes, out, out_raw, flags, stream
    assert ragged(FAKE, 0, None, FAKE, None, 8, 16, FAKE, ws, FAKE, None, 0, None) == 1
    assert ragged(FAKE, 0, None, FAKE, FAKE, 8, 4096, FAKE, ws, FAKE, None, 0, None) == 3
    assert ragged(FAKE, 0, None, FAKE, FAKE, 8, 16, None, ws, FAKE, None, 0, None) == 5
    assert ragged(FAKE, 0, None, FAKE, FAKE, 8, 16, FAKE, ws, FAKE, None, 3, None) == 1
    packed = lib.topk_transform_paged_packed
    # scores, stride, row_starts, seq_lens, page_table, pt_stride, page_size, pt_row_starts, row_to_batch,
    # batch, k, ws, ws_bytes, out, out_raw, flags, stream
    assert packed(FAKE, 64, None, FAKE, FAKE, 4, 64, FAKE, FAKE, 8, 0, FAKE, ws, FAKE, None, 0, None) == 3
    assert packed(FAKE, 64, None, FAKE, FAKE, 4, 48, FAKE, FAKE, 8, 16, FAKE, ws, FAKE, None, 0, None) == 4
    assert packed(FAKE, 64, None, FAKE, None, 4, 64, FAKE, FAKE, 8, 16, FAKE, ws, FAKE, None, 0, None) == 1
    assert packed(FAKE_UNALIGNED, 64, None, FAKE, FAKE, 4, 64, FAKE, FAKE, 8, 16, FAKE, ws, FAKE, None, 0, None) == 2
    assert packed(FAKE, 64, None, FAKE, FAKE, 4, 64, FAKE, FAKE, 8, 16, FAKE, ws - 1, FAKE, None, 0, None) == 5
    assert packed(FAKE, 64, None, FAKE, FAKE, 4, 64, None, None, 8, 16, FAKE, ws, FAKE, None, 4, None) == 1
    assert packed(None, 0, None, None, None, 0, 1, None, None, 0, 16, FAKE, lib.topk_workspace_bytes(0),
                  None, None, 0, None) == 0
    # an empty batch is a no-op that enqueues nothing
    assert ragged(None, 0, None, None, None, 0, 16, FAKE, lib.topk_workspace_bytes(0), None, None, 0, None) == 0
    assert paged(None, 0, None, None, None, 0, 1, 0, 16, FAKE, lib.topk_workspace_bytes(0), None, None, 0, None) == 0


def test_swa_transform_validation(lib):
    ws = lib.topk_workspace_bytes(8)
    swa = lib.topk_transform_ragged_swa
    # scores, stride, row_starts, seq_lens, out_offsets, batch, k, ws, ws_bytes, positions, window,
    # swa_offsets, out_width, out, out_raw, flags, stream
    assert swa(FAKE, 0, None, FAKE, FAKE, 8, 16, FAKE, ws, None, 4, None, 20, FAKE, None, 0, None) == 1  # no positions
    assert swa(FAKE, 0, None, FAKE, None, 8, 16, FAKE, ws, FAKE, 4, None, 20, FAKE, None, 0, None) == 1  # no offsets
    assert swa(FAKE, 0, None, FAKE, FAKE, 8, 16, FAKE, ws, FAKE, -1, None, 20, FAKE, None, 0, None) == 1
    assert swa(FAKE, 0, None, FAKE, FAKE, 8, 16, FAKE, ws, FAKE, (1 << 20) + 1, None, 1 << 21, FAKE, None, 0,
               None) == 1
    assert swa(FAKE, 0, None, FAKE, FAKE, 8, 16, FAKE, ws, FAKE, 4, None, 19, FAKE, None, 0, None) == 1  # too narrow
    assert swa(FAKE, 0, None, FAKE, FAKE, 8, 0, FAKE, ws, FAKE, 4, None, 20, FAKE, None, 0, None) == 3
    assert swa(FAKE, 0, None, FAKE, FAKE, 8, 16, FAKE, ws - 1, FAKE, 4, None, 20, FAKE, None, 0, None) == 5
    assert swa(FAKE, 0, None, FAKE, FAKE, 8, 16, FAKE, ws, FAKE, 4, None, 20, FAKE, None, 2, None) == 1
    assert swa(None, 0, None, None, None, 0, 16, FAKE, lib.topk_workspace_bytes(0), None, 4, None, 20, None, None,
               0, None) == 0


def test_indexer_logits_validation(lib):
    fn = lib.topk_indexer_logits
    # q, kv, kv_scale, weights, ks, ke, n_q, n_kv, logits, stride, device_flags, stream
    assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1, 10, FAKE, 16, FAKE, None) == 1
    assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, -1, FAKE, 16, FAKE, None) == 1
    assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, (1 << 24) + 1, 10, FAKE, 16, FAKE, None) == 1
    assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, (1 << 30) - 255, FAKE, 16, FAKE, None) == 1
    assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, FAKE, -16, FAKE, None) == 1
    assert fn(None, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, FAKE, 16, FAKE, None) == 1
    assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, 10, FAKE, 16, FAKE, None) == 1
    assert fn(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, FAKE, 16, None, None) == 1  # no flag word
    assert fn(FAKE_UNALIGNED, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 10, FAKE, 16, FAKE, None) == 2
    assert fn(FAKE, FAKE_UNALIGNED, FAKE, FAKE, FAKE, FAKE, 4, 10, FAKE, 16, FAKE, None) == 2
    assert fn(FAKE, FAKE, FAKE, FAKE_UNALIGNED, FAKE, FAKE, 4, 10, FAKE, 16, FAKE, None) == 2  # weights
    # nothing to compute: no-ops that enqueue nothing
    assert fn(None, None, None, None, None, None, 0, 10, None, 0, None, None) == 0
    assert fn(None, None, None, None, None, None, 4, 0, None, 0, None, None) == 0


def test_status_strings(lib):
    for s in range(7):
        assert lib.topk_status_string(s)
    assert lib.topk_status_string(99) == b"unknown status"


def test_read_errors_validation(lib):
    assert lib.topk_read_device_errors(None, None, None, None) == 1
