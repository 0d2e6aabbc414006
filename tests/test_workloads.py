"""The seeded input generators keep the recipes the benchmark and the parity
tests rely on: the same seed gives the same bytes, windows hold the stated
values and only the 1e3 sentinel lies outside them, page tables are
permutations, and the per-row arrays follow the stated formulas. CPU only,
on scaled-down sizes."""

from __future__ import annotations

import numpy as np
import torch

from sparse_attention_top_row_gb300 import workloads as wl

SENT = np.float32(wl.SENTINEL)


def _np(x):
    return None if x is None else x.detach().cpu().numpy()


def _inside_mask(w):
    """[B, stride] mask of the window positions (stride > 0 workloads)."""
    B, stride = int(w["batch"]), int(w["score_stride"])
    starts = _np(w["row_starts"]) if w.get("row_starts") is not None else np.zeros(B, np.int64)
    lens = _np(w["seq_lens"])
    cols = np.arange(stride)[None, :]
    return (cols >= starts[:, None]) & (cols < (starts + lens)[:, None])


def _same_bytes(a, b):
    for key in a:
        if isinstance(a[key], torch.Tensor):
            assert torch.equal(a[key], b[key]), key


def test_generators_are_deterministic():
    _same_bytes(wl.ragged_tiny("cpu", sub_id=3), wl.ragged_tiny("cpu", sub_id=3))
    _same_bytes(wl.paged_decode("cpu", batch=4, seq_len=512), wl.paged_decode("cpu", batch=4, seq_len=512))
    a = wl.paged_decode("cpu", sub_id=0, batch=4, seq_len=512)
    b = wl.paged_decode("cpu", sub_id=1, batch=4, seq_len=512)
    assert not torch.equal(a["scores"], b["scores"])


def test_ragged_tiny_recipe():
    w = wl.ragged_tiny("cpu", sub_id=0)
    lens, starts = _np(w["seq_lens"]), _np(w["row_starts"])
    assert w["score_stride"] == 0 and np.all((lens >= 1) & (lens <= 4096))
    np.testing.assert_array_equal(starts, np.concatenate([[0], np.cumsum(lens)[:-1]]))
    np.testing.assert_array_equal(_np(w["out_offsets"]), starts)
    s = _np(w["scores"])
    end = int(lens.sum())
    assert np.all(s[end:] == SENT) and not np.any(s[:end] == SENT)
    assert (s.size - end) >= 64 and s.size % 4 == 0


def test_paged_decode_recipe():
    w = wl.paged_decode("cpu", batch=6, seq_len=1024, k=100, page_size=64)
    assert np.all(_np(w["seq_lens"]) == 1024) and w["row_starts"] is None
    pt = _np(w["page_table"])
    assert pt.shape == (6, 16)
    np.testing.assert_array_equal(np.sort(pt.reshape(-1)), np.arange(6 * 16))


def test_ragged_extend_recipe():
    w = wl.ragged_extend("cpu", chunk=1, rows_per_chunk=8, n_req=2, prefix=100, new=12, k=10)
    rows = np.arange(8, 16)
    np.testing.assert_array_equal(_np(w["seq_lens"]), 100 + rows % 12 + 1)
    np.testing.assert_array_equal(_np(w["row_starts"]), (rows // 12) * 112)
    np.testing.assert_array_equal(_np(w["out_offsets"]), _np(w["row_starts"]))
    s = _np(w["scores"]).reshape(8, -1)
    inside = _inside_mask(w)
    assert np.all(s[~inside] == SENT) and not np.any(s[inside] == SENT)
    outliers = np.mean(s[inside] == np.float32(4.0))
    assert 0.0 < outliers < 0.05


def test_paged_long_values_are_bf16():
    w = wl.paged_long("cpu", batch=2, seq_len=4096, k=64)
    bits = _np(w["scores"]).view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0)
    np.testing.assert_array_equal(np.sort(_np(w["page_table"]).reshape(-1)), np.arange(2 * 64))


def test_mixed_recipe():
    k = 64
    for mode in ("paged", "ragged"):
        w = wl.mixed("cpu", mode=mode, k=k, batch=12, max_len=20000, min_len=16)
        lens = _np(w["seq_lens"])
        expect = [min(x, 20000) for x in wl.boundary_lengths(k)]
        np.testing.assert_array_equal(lens[:9], expect)
        assert np.all((lens >= 16) & (lens <= 20000))
        s = _np(w["scores"]).reshape(12, -1)
        inside = _inside_mask(w)
        assert np.all(s[~inside] == SENT) and not np.any(s[inside] == SENT)
        if mode == "ragged":
            starts = _np(w["row_starts"])
            assert np.all((starts >= 0) & (starts < 4))
            np.testing.assert_array_equal(_np(w["out_offsets"]), np.arange(12) * w["score_stride"] + starts)


def test_paged_packed_recipe():
    w = wl.paged_packed("cpu", n_req=3, q_rows=4, min_tokens=500, max_tokens=900, window=300, k=50, page_size=16)
    ptrs, rtb = _np(w["page_table_row_starts"]), _np(w["row_to_batch"])
    lens, starts = _np(w["seq_lens"]), _np(w["row_starts"])
    np.testing.assert_array_equal(rtb, np.repeat(np.arange(3), 4))
    s = _np(w["scores"]).reshape(12, -1)
    for r in range(3):
        rows = np.nonzero(rtb == r)[0]
        # the request's keys occupy one block of columns in every one of its rows
        cols = np.nonzero(s[rows[0]] != SENT)[0]
        a, e = int(cols[0]), int(cols[-1]) + 1
        tokens = e - a
        assert len(cols) == tokens
        for j, b in enumerate(rows):
            tok = tokens - 4 + j                                  # the query's own token
            assert ptrs[b] == max(0, tok + 1 - 300) and lens[b] == tok + 1 - ptrs[b]
            assert starts[b] == a + ptrs[b]
    assert np.all(np.sort(_np(w["page_table"]).reshape(-1)) == np.arange(_np(w["page_table"]).size))
