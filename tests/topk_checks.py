"""Checks shared by the oracle pins and the GPU parity tests.

Everything here is written independently of the oracle's C++: the brute force
ranks by numeric value with the sign of zero as a second key (no bit tricks),
and the page-table check expands the table into a full logical→physical map
instead of dividing positions.
"""

from __future__ import annotations

import numpy as np


def host(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        return x.detach().cpu().numpy()
    return np.asarray(x)


# --------------------------------------------------------------------------
# brute force: an element is selected iff fewer than k elements rank above it
# --------------------------------------------------------------------------

def brute_force_select(values, k):
    """values: [R, n] float array (no NaN). Returns a bool [R, n] mask of the
    top-k under the order (value, sign of zero) with ties to the lowest
    position. O(n^2) rank counting, independent of any sort."""
    v = np.asarray(values, dtype=np.float64)
    s = np.copysign(1.0, v)
    vp, vq = v[:, :, None], v[:, None, :]
    sp, sq = s[:, :, None], s[:, None, :]
    beats = (vq > vp) | ((vq == vp) & (sq > sp))          # [R, p, q]: q ranks above p
    same = (vq == vp) & (sq == sp)
    n = v.shape[1]
    lower_pos = np.arange(n)[None, :] < np.arange(n)[:, None]  # [p, q]: q < p
    rank = beats.sum(2) + (same & lower_pos[None]).sum(2)
    return rank < k


def expand_page_table(page_table_row, page_size, length):
    """Logical position -> physical slot for one row, by expanding each page
    into its page_size consecutive slots."""
    pages = np.asarray(page_table_row, dtype=np.int64)
    slots = (pages[:, None] * page_size + np.arange(page_size)[None, :]).reshape(-1)
    return slots[:length]


# --------------------------------------------------------------------------
# per-row views of a workload
# --------------------------------------------------------------------------

class HostWorkload:
    """Host copies of a workload's arrays with per-row helpers."""

    def __init__(self, w):
        self.w = w
        self.mode = w["mode"]
        self.k = int(w["k"])
        self.stride = int(w["score_stride"])
        self.scores = host(w["scores"]).reshape(-1)
        self.seq_lens = host(w["seq_lens"]).astype(np.int64)
        rs = w.get("row_starts")
        self.row_starts = None if rs is None else host(rs).astype(np.int64)
        oo = w.get("out_offsets")
        self.out_offsets = None if oo is None else host(oo).astype(np.int64)
        pt = w.get("page_table")
        self.page_table = None if pt is None else host(pt).reshape(-1).astype(np.int64)
        self.pt_stride = int(w.get("page_table_stride", 0))
        ptrs = w.get("page_table_row_starts")
        self.pt_row_starts = None if ptrs is None else host(ptrs).astype(np.int64)
        rtb = w.get("row_to_batch")
        self.row_to_batch = None if rtb is None else host(rtb).astype(np.int64)
        self.page_size = int(w.get("page_size", 1))
        self.batch = int(w["batch"])

    def start(self, b):
        return 0 if self.row_starts is None else int(self.row_starts[b])

    def length(self, b):
        L = int(self.seq_lens[b])
        bad_table_start = self.pt_row_starts is not None and int(self.pt_row_starts[b]) < 0
        return 0 if (L < 0 or self.start(b) < 0 or bad_table_start) else L

    def window(self, b):
        base = b * self.stride + self.start(b)
        return self.scores[base:base + self.length(b)]

    def transform(self, b, raw):
        raw = np.asarray(raw, dtype=np.int64)
        if self.mode == "paged":
            # packed rows: table row row_to_batch[b], tokens from page_table_row_starts[b]
            t = b if self.row_to_batch is None else int(self.row_to_batch[b])
            t0 = 0 if self.pt_row_starts is None else int(self.pt_row_starts[b])
            row = self.page_table[t * self.pt_stride:(t + 1) * self.pt_stride]
            phys = expand_page_table(row, self.page_size, t0 + max(self.length(b), 1))
            return phys[t0 + raw]
        return raw + self.out_offsets[b]


def bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def order_keys(x):
    """Unsigned keys in the selection order (used only to compare GPU output
    with the oracle's; the pins rank with brute_force_select instead)."""
    b = bits(x).astype(np.uint64)
    neg = (b >> 31) == 1
    return np.where(neg, (~b) & 0xFFFFFFFF, b | 0x80000000).astype(np.uint64)


def check_row_invariants(hw: HostWorkload, b, out_row, raw_row, sentinel=1.0e3):
    """Invariants every correct output row satisfies (any tie choice)."""
    k = hw.k
    L = hw.length(b)
    raw_row = np.asarray(raw_row, dtype=np.int64)
    out_row = np.asarray(out_row, dtype=np.int64)
    sel = raw_row[raw_row >= 0]
    n = min(k, L)
    assert sel.size == n, f"row {b}: {sel.size} selected, expected min(k, L) = {n}"
    assert np.count_nonzero(raw_row == -1) == k - n, f"row {b}: wrong -1 padding count"
    assert np.all(out_row[raw_row < 0] == -1), f"row {b}: padding is not -1"
    assert np.unique(sel).size == sel.size, f"row {b}: duplicate positions"
    assert np.all((sel >= 0) & (sel < L)), f"row {b}: position outside the window"
    np.testing.assert_array_equal(out_row[raw_row >= 0], hw.transform(b, raw_row[raw_row >= 0]),
                                  err_msg=f"row {b}: transform mismatch")
    if L > k:
        win = hw.window(b)
        keys = order_keys(win)
        mask = np.zeros(L, dtype=bool)
        mask[sel] = True
        assert keys[mask].min() >= keys[~mask].max(), f"row {b}: an unselected score beats a selected one"
        # the sentinel lives only outside windows; nothing selected may equal it
        # unless the window itself holds that value
        if not np.any(win == sentinel):
            assert not np.any(win[sel] == sentinel)


def compare_with_oracle(hw: HostWorkload, out, out_raw, ref_out, ref_raw, rows=None, deterministic=True):
    """GPU rows vs oracle rows.

    deterministic: sorted output rows (and raw rows) bit-exact.
    default mode: the selected score multisets are bit-identical, so the index
    sets differ only by swaps of equal scores; every output is still checked
    against the transform and the invariants.
    """
    out = np.asarray(out)
    out_raw = np.asarray(out_raw)
    rows = range(hw.batch) if rows is None else rows
    for i, b in enumerate(rows):
        o, r = out[i], out_raw[i]
        ro, rr = ref_out[i], ref_raw[i]
        check_row_invariants(hw, b, o, r)
        if deterministic:
            np.testing.assert_array_equal(np.sort(r), np.sort(rr), err_msg=f"row {b}: raw positions differ")
            np.testing.assert_array_equal(np.sort(o), np.sort(ro), err_msg=f"row {b}: outputs differ")
        else:
            win = hw.window(b)
            ours = np.sort(bits(win[r[r >= 0]]))
            refs = np.sort(bits(win[rr[rr >= 0]]))
            np.testing.assert_array_equal(ours, refs, err_msg=f"row {b}: selected score multisets differ")
