"""The benchmark's roofline numerator (algorithmic bytes per launch), counted
by hand on small cases: 4 B per score of every non-trivial row, 4 B per
output slot, 4 B per per-row array read, and 4 B per distinct page-table
entry the selected positions touch (packed rows: counted at their
page-table start). Also the end-to-end leg's packed input copy. CPU only."""

from __future__ import annotations

import torch

import bench
from sparse_attention_top_row_gb300 import workloads as wl


def test_ragged_bytes():
    w = wl.custom("ragged", 4, [[1.0] * 10, [2.0] * 3, [0.5] * 7], row_starts=[0, 1, 2], out_offsets=[0, 0, 0])
    raw = torch.full((3, 4), -1, dtype=torch.int32)
    # rows 0 and 2 are non-trivial (10 and 7 > k = 4); row 1 is trivial (3 <= 4)
    scores = 4 * (10 + 7)
    out = 4 * 4 * 3
    meta = 4 * 3 * 3  # seq_lens, row_starts, out_offsets
    assert bench.algorithmic_bytes(w, raw) == scores + out + meta


def test_paged_bytes_count_distinct_pages():
    w = wl.custom("paged", 3, [[float(i) for i in range(12)]], page_size=4, seed=1)
    raw = torch.tensor([[0, 5, 6]], dtype=torch.int32)  # pages 0, 1, 1: two distinct entries
    assert bench.algorithmic_bytes(w, raw) == 4 * 12 + 4 * 3 + 4 * 1 + 4 * 2


def test_packed_bytes_count_pages_from_the_table_start():
    w = wl.custom("paged", 3, [[float(i) for i in range(12)]], page_size=4, seed=1)
    w["page_table"] = torch.arange(16, dtype=torch.int32).view(2, 8)
    w["page_table_stride"] = 8
    w["page_table_row_starts"] = torch.tensor([3], dtype=torch.int32)
    w["row_to_batch"] = torch.tensor([1], dtype=torch.int32)
    raw = torch.tensor([[0, 1, 5]], dtype=torch.int32)  # tokens 3, 4, 8: pages 0, 1, 2
    assert bench.algorithmic_bytes(w, raw) == 4 * 12 + 4 * 3 + 4 * 3 + 4 * 3


def test_e2e_inputs_pack_into_one_copy(monkeypatch):
    """The end-to-end leg copies a launch's inputs as one packed buffer: every
    tensor comes back bit for bit from its 256-byte-aligned slot."""
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)   # no CUDA here
    for w in (wl.paged_decode("cpu", batch=8, seq_len=1024, k=64), wl.ragged_tiny("cpu"),
              wl.paged_packed("cpu", n_req=2, q_rows=2, min_tokens=500, max_tokens=900, window=300, k=50,
                              page_size=16)):
        host, dev, dw = bench.packed_inputs(w, "cpu")
        dev.copy_(host)
        payload = 0
        for key, v in w.items():
            if isinstance(v, torch.Tensor):
                payload += v.numel() * v.element_size()
                assert dw[key].dtype == v.dtype and torch.equal(dw[key], v), key
                assert (dw[key].data_ptr() - dev.data_ptr()) % 256 == 0 and dw[key].is_contiguous()
        assert payload <= host.numel() < payload + 256 * len(w)


def test_logits_flops_count_window_pairs():
    """The indexer logits' roofline numerator: 2 * 64 * 128 FLOPs per (query,
    key) pair inside a window, windows clamped to [0, n_kv), empty and
    reversed windows counting nothing."""
    w = dict(ks=torch.tensor([0, -5, 90, 40, 7], dtype=torch.int32),
             ke=torch.tensor([10, 3, 130, 40, 2], dtype=torch.int32), n_kv=100)
    pairs = 10 + 3 + 10 + 0 + 0
    assert bench.logits_flops(w) == pairs * 2 * 64 * 128
