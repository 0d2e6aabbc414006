"""Property-based pins of the CPU oracle (hypothesis; CPU only).

The scores are arbitrary fp32 bit patterns: NaNs with any sign and payload
(quiet or signalling), infinities, subnormals, signed zeros and ordinary
values, mixed with a small alphabet so that equal scores are common. The
expected selection comes from brute-force rank counting under the IEEE 754
totalOrder predicate (IEEE 754-2008, 5.10), written here by case analysis on
sign, NaN-ness and payload rather than through a bit-pattern key: a score at
position p is kept iff fewer than k scores of its window rank above it, where
q ranks above p when x_q is after x_p in totalOrder, or when they are the same
datum and q < p (ties to the lowest position). That is the order the pages'
fp32 -> uint32 key map induces, so any slip in the oracle's key map, tie rule,
window start, page-table lookup (plain or packed) or padding shows up here.
The scores go to the oracle as raw bits (never through Python floats, which
would quiet signalling NaNs).
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from topk_checks import HostWorkload

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies
given, settings = hypothesis.given, hypothesis.settings

_ALPHABET = [0x00000000, 0x80000000, 0x3F800000, 0xBF800000, 0x7F800000, 0xFF800000,  # 0, -0, 1, -1, inf, -inf
             0x7FC00000, 0xFFC00000, 0x7F800001, 0x00000001, 0x80000001, 0x7F7FFFFF]  # NaNs, subnormals, max


def _is_nan(u):
    return (u & 0x7F800000) == 0x7F800000 and (u & 0x007FFFFF) != 0


def _value(u):
    return float(np.array([u], dtype=np.uint32).view(np.float32)[0])


def total_order_above(uq, up):
    """True when the fp32 datum with bits uq comes strictly after the one with
    bits up in IEEE 754 totalOrder."""
    sq, sp = uq >> 31, up >> 31
    nq, np_ = _is_nan(uq), _is_nan(up)
    if nq or np_:
        if nq and np_:
            if sq != sp:
                return sp == 1                       # -NaN < +NaN
            pq, pp = uq & 0x007FFFFF, up & 0x007FFFFF
            return pq > pp if sq == 0 else pq < pp   # a negative NaN with a larger payload is lower
        if nq:
            return sq == 0                           # +NaN above every number, -NaN below
        return sp == 1
    vq, vp = _value(uq), _value(up)
    if vq != vp:
        return vq > vp
    if vq == 0.0:                                    # -0 < +0
        return math.copysign(1.0, vq) > math.copysign(1.0, vp)
    return False


def brute_force_positions(window_bits, k):
    n = len(window_bits)
    keep = []
    for p in range(n):
        rank = 0
        for q in range(n):
            if q == p:
                continue
            if total_order_above(window_bits[q], window_bits[p]):
                rank += 1
            elif q < p and window_bits[q] == window_bits[p]:
                rank += 1
        if rank < k:
            keep.append(p)
    return np.asarray(keep, dtype=np.int64)


bit_patterns = st.one_of(st.integers(0, 0xFFFFFFFF), st.sampled_from(_ALPHABET))


@st.composite
def workloads(draw):
    mode = draw(st.sampled_from(["ragged", "paged"]))
    k = draw(st.integers(1, 24))
    rows = draw(st.lists(st.lists(bit_patterns, min_size=0, max_size=20), min_size=1, max_size=5))
    B = len(rows)
    starts = [draw(st.integers(0, 5)) for _ in range(B)]
    stride = (max(s + len(r) for s, r in zip(starts, rows)) + 3) // 4 * 4 + 4 * draw(st.integers(0, 2))
    sentinel = int(np.array([1.0e3], dtype=np.float32).view(np.uint32)[0])
    buf = np.full(B * stride + 64, sentinel, dtype=np.uint32)
    for b, (s, r) in enumerate(zip(starts, rows)):
        buf[b * stride + s:b * stride + s + len(r)] = np.asarray(r, dtype=np.uint32)
    w = dict(name="hypothesis", mode=mode, k=k, batch=B, score_stride=stride,
             scores=torch.from_numpy(buf.view(np.float32)),
             seq_lens=torch.tensor([len(r) for r in rows], dtype=torch.int32),
             row_starts=torch.tensor(starts, dtype=torch.int32))
    if mode == "paged":
        ps = draw(st.sampled_from([1, 2, 4, 8, 16]))
        packed = draw(st.booleans())                 # request-local table starts, shared table rows
        t0 = [draw(st.integers(0, 6)) if packed else 0 for _ in range(B)]
        pages = max((stride + 6 + ps - 1) // ps, 1)
        perm = draw(st.permutations(list(range(B * pages))))
        w.update(page_size=ps, page_table=torch.tensor(perm, dtype=torch.int32).view(B, pages),
                 page_table_stride=pages, out_offsets=None)
        if packed:
            w.update(page_table_row_starts=torch.tensor(t0, dtype=torch.int32),
                     row_to_batch=torch.tensor([draw(st.integers(0, B - 1)) for _ in range(B)],
                                               dtype=torch.int32))
    else:
        offs = [draw(st.integers(-(1 << 20), 1 << 20)) for _ in range(B)]
        w.update(page_size=1, page_table=None, page_table_stride=0,
                 out_offsets=torch.tensor(offs, dtype=torch.int32))
    return w, rows


@settings(max_examples=300, deadline=None, derandomize=True)
@given(workloads())
def test_oracle_matches_total_order_brute_force(case):
    w, rows = case
    hw = HostWorkload(w)
    out, raw, err = oracle.run_workload(w)
    assert err == 0
    for b, r in enumerate(rows):
        expect = brute_force_positions([int(u) for u in r], hw.k)
        got = raw[b][raw[b] >= 0]
        np.testing.assert_array_equal(np.sort(got), expect, err_msg=f"row {b}")
        np.testing.assert_array_equal(np.sort(out[b][raw[b] >= 0]), np.sort(hw.transform(b, expect)))
        assert np.all(out[b][raw[b] < 0] == -1) and np.all(raw[b][raw[b] < 0] == -1)
        assert int((raw[b] >= 0).sum()) == min(hw.k, len(r))


def test_total_order_reference_points():
    """The comparator itself on points totalOrder fixes."""
    order = [0xFFC00001, 0xFFC00000, 0xFF800000, 0xFF7FFFFF, 0xBF800000, 0x80000001, 0x80000000,
             0x00000000, 0x00000001, 0x3F800000, 0x7F7FFFFF, 0x7F800000, 0x7F800001, 0x7FC00000]
    for i, a in enumerate(order):
        for j, b in enumerate(order):
            assert total_order_above(b, a) == (j > i), (hex(a), hex(b))
