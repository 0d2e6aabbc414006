"""Pins of the CPU oracle to things other than itself (no GPU needed).

* hand-built examples worked from the pages' definitions (tests/golden/);
* brute-force rank counting on random tiny rows, both modes;
* an exhaustive sweep of short vectors over {-1, -0.0, 0.0, 1, 2} (ties and
  signed zeros) for every k up to the length;
* numpy.partition on tie-free rows (a library routine on a special case);
* an independent page-table expansion for the PAGED transform;
* invariants on scaled-down versions of every workload shape;
* the indexer logits: every E4M3 code against torch's float8_e4m3fn, a
  hand-worked example and a closed form at the 64 x 128 head shape;
* planted mistakes in the oracle (compiled variants) are each caught.
"""

from __future__ import annotations

import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_top_row_gb300 import workloads as wl
from topk_checks import HostWorkload, brute_force_select, check_row_invariants, expand_page_table

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _golden_workload(case):
    mode = case["mode"]
    if "buffer" in case:
        buf = np.asarray(case["buffer"], dtype=np.float32)
        return dict(mode=mode, k=case["k"], scores=torch.from_numpy(buf),
                    score_stride=case["score_stride"],
                    row_starts=torch.tensor(case["row_starts"], dtype=torch.int32),
                    seq_lens=torch.tensor(case["seq_lens"], dtype=torch.int32),
                    out_offsets=torch.tensor(case["out_offsets"], dtype=torch.int32),
                    page_table=None, page_table_stride=0, page_size=1,
                    batch=len(case["seq_lens"]), name=case["name"])
    w = wl.custom(mode, case["k"], case["rows"], page_size=case.get("page_size", 1),
                  page_table=case.get("page_table"))
    for key in ("page_table_row_starts", "row_to_batch"):  # packed PAGED cases
        if key in case:
            w[key] = torch.tensor(case[key], dtype=torch.int32)
    return w


def golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


# ------------------------------------------------------------------ pin families

def pin_golden(mutant=0):
    for case in golden_cases():
        w = _golden_workload(case)
        out, raw, _ = oracle.run_workload(w, mutant=mutant)
        assert np.sort(out, axis=1).tolist() == case["det"], case["name"]
        assert np.sort(raw, axis=1).tolist() == case["det_raw"], case["name"]


def pin_bruteforce(mutant=0, seed=1, n_rows=300):
    rng = np.random.default_rng(seed)
    for trial in range(6):
        mode = "paged" if trial % 2 else "ragged"
        k = int(rng.choice([1, 2, 3, 5, 8, 16, 33, 64]))
        rows, starts = [], []
        for _ in range(n_rows // 6):
            L = int(rng.integers(0, 65))
            if trial % 3 == 0:
                vals = rng.choice([-2.0, -1.0, -0.0, 0.0, 0.5, 1.0, 3.0], size=L)
            else:
                vals = rng.standard_normal(L).astype(np.float32)
            rows.append([float(v) for v in vals])
            starts.append(int(rng.integers(0, 7)))
        offs = [int(x) for x in rng.integers(-5, 1000, size=len(rows))]
        ps = int(rng.choice([1, 2, 4, 8]))
        w = wl.custom(mode, k, rows, row_starts=starts, out_offsets=offs, page_size=ps,
                      seed=seed + trial)
        hw = HostWorkload(w)
        out, raw, err = oracle.run_workload(w, mutant=mutant)
        assert err == 0
        for b, r in enumerate(rows):
            L = len(r)
            if L == 0:
                expect = np.zeros(0, dtype=np.int64)
            else:
                expect = np.nonzero(brute_force_select(np.asarray([hw.window(b)]), k)[0])[0]
            got = raw[b][raw[b] >= 0]
            np.testing.assert_array_equal(np.sort(got), expect, err_msg=f"trial {trial} row {b}")
            np.testing.assert_array_equal(np.sort(out[b][raw[b] >= 0]), np.sort(hw.transform(b, expect)))
            assert np.all(out[b][raw[b] < 0] == -1)


def pin_exhaustive(mutant=0, max_n=8):
    alphabet = np.array([-1.0, -0.0, 0.0, 1.0, 2.0], dtype=np.float32)
    for n in range(1, max_n + 1):
        combos = np.array(list(itertools.product(range(len(alphabet)), repeat=n)), dtype=np.int64)
        vals = alphabet[combos]                      # [R, n]
        R = vals.shape[0]
        scores = np.ascontiguousarray(vals.reshape(-1))
        seq_lens = np.full(R, n, dtype=np.int32)
        offs = np.zeros(R, dtype=np.int32)
        for k in range(1, n + 1):
            out, raw, _ = oracle.topk_transform(oracle.RAGGED, scores, n, None, seq_lens, k,
                                                out_offsets=offs, mutant=mutant)
            expect = brute_force_select(vals, k)
            got = np.zeros((R, n), dtype=bool)
            rows = np.repeat(np.arange(R), k)
            sel = raw.reshape(-1)
            valid = sel >= 0
            got[rows[valid], sel[valid]] = True
            bad = np.nonzero((got != expect).any(1))[0]
            assert bad.size == 0, f"n={n} k={k}: first bad row {vals[bad[0]].tolist()}"


def pin_partition(mutant=0, seed=3):
    rng = np.random.default_rng(seed)
    for L, k in [(100, 7), (1000, 100), (5000, 2048), (3000, 1)]:
        # distinct magnitudes with random signs
        x = np.stack([rng.permutation(np.arange(1, L + 1)) * rng.choice([-1.0, 1.0], size=L) / 64.0
                      for _ in range(4)]).astype(np.float32)
        # tie-free and no zeros: the special case where plain numeric order is the order
        assert all(np.unique(r).size == L for r in x) and not np.any(x == 0)
        out, raw, _ = oracle.topk_transform(oracle.RAGGED, x.reshape(-1), L, None,
                                            np.full(4, L, np.int32), k,
                                            out_offsets=np.zeros(4, np.int32), mutant=mutant)
        for b in range(4):
            kth = -np.partition(-x[b], k - 1)[k - 1]            # k-th largest, by library routine
            expect = np.nonzero(x[b] >= kth)[0]
            np.testing.assert_array_equal(np.sort(raw[b]), expect)


def pin_paged_expansion(mutant=0, seed=4):
    for ps in (1, 2, 64, 256):
        w = wl.custom("paged", 37, [list(np.random.default_rng(seed + ps).standard_normal(700))
                                   for _ in range(5)], page_size=ps, seed=ps)
        out, raw, _ = oracle.run_workload(w, mutant=mutant)
        pt = w["page_table"].numpy()
        for b in range(5):
            phys = expand_page_table(pt[b], ps, 700)
            np.testing.assert_array_equal(out[b], phys[raw[b]])
            # inverting the table maps every physical slot back to its position
            inv = {int(s): p for p, s in enumerate(phys)}
            assert [inv[int(s)] for s in out[b]] == raw[b].tolist()


def pin_packed_expansion(mutant=0, seed=9):
    """Packed PAGED rows: each output is the request table, expanded slot by
    slot, read at page_table_row_starts + p (an expansion written here, not
    the oracle's division); with both arrays absent the plain PAGED result."""
    for ps in (1, 16, 64):
        w = wl.paged_packed("cpu", sub_id=ps, n_req=3, q_rows=3, min_tokens=600, max_tokens=1500,
                            window=700, k=50, page_size=ps)
        out, raw, err = oracle.run_workload(w, mutant=mutant)
        assert err == 0
        pt = w["page_table"].numpy()
        ptrs, rtb = w["page_table_row_starts"].numpy(), w["row_to_batch"].numpy()
        for b in range(w["batch"]):
            phys = expand_page_table(pt[rtb[b]], ps, int(ptrs[b]) + int(w["seq_lens"][b]))
            np.testing.assert_array_equal(out[b], phys[int(ptrs[b]) + raw[b]])
        plain = dict(w, page_table_row_starts=None, row_to_batch=None)
        plain["page_table"] = w["page_table"][w["row_to_batch"].long()]
        out2, raw2, _ = oracle.run_workload(plain, mutant=mutant)
        np.testing.assert_array_equal(raw2, raw)
        if ps == 1:  # token t of a request is slot pt[r][t]: shifting the start shifts the slots
            for b in range(w["batch"]):
                np.testing.assert_array_equal(out[b], pt[rtb[b]][int(ptrs[b]) + raw[b]])


def pin_invariants(mutant=0):
    cases = [
        wl.ragged_tiny("cpu", sub_id=0),
        wl.paged_decode("cpu", batch=8, seq_len=2048, k=256),
        wl.ragged_extend("cpu", chunk=0, rows_per_chunk=16, n_req=2, prefix=1000, new=24, k=200),
        wl.paged_long("cpu", batch=2, seq_len=8192, k=512),
        wl.mixed("cpu", mode="ragged", k=64, batch=12, max_len=4000, min_len=16),
        wl.mixed("cpu", mode="paged", k=64, batch=12, max_len=4000, min_len=16),
        wl.paged_packed("cpu", n_req=2, q_rows=3, min_tokens=500, max_tokens=2000, window=900, k=100),
    ]
    for w in cases:
        hw = HostWorkload(w)
        before = hw.scores.copy()
        out, raw, err = oracle.run_workload(w, mutant=mutant)
        assert err == 0
        for b in range(hw.batch):
            check_row_invariants(hw, b, out[b], raw[b])
        np.testing.assert_array_equal(hw.scores.view(np.uint32), before.view(np.uint32))


PINS = [pin_golden, pin_bruteforce, pin_exhaustive, pin_partition, pin_paged_expansion, pin_packed_expansion,
        pin_invariants]


SWA_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "swa_examples.json")


def pin_swa_golden(mutant=0):
    """The SWA combine's hand-built examples (tests/golden/swa_examples.json)."""
    with open(SWA_GOLDEN) as f:
        g = json.load(f)
    w = wl.custom("ragged", g["k"], g["rows"], out_offsets=g["out_offsets"])
    w["seq_lens"] = torch.tensor(g["seq_lens"], dtype=torch.int32)
    out, raw, _ = oracle.run_workload(w, mutant=mutant)
    res = oracle.swa_combine(out, raw, g["positions"], g["window_size"], g["swa_offsets"], g["width"],
                             mutant=mutant)
    for case in g["cases"]:
        row = res[case["row"]]
        n = len(case["topk_sorted"])
        assert sorted(row[:n].tolist()) == case["topk_sorted"], case["why"]
        assert row[n:].tolist() == case["tail"], case["why"]


def pin_swa_formula(mutant=0, seed=11):
    """On compressed rows of L = (pos + 1) // ratio entries, the combined row
    carries min((pos + 1) // ratio, k) selected entries (the page's topk_len),
    exactly the row's top-k selection; its window part is the set of tokens t
    with 0 <= t <= pos and pos - t < window (a brute-force filter of 0..pos),
    plus the row's SWA offset, in ascending order; the rest is -1."""
    rng = np.random.default_rng(seed)
    for ratio, window, k in ((4, 8, 5), (1, 3, 16), (128, 16, 2)):
        B = 12
        pos = rng.integers(-1, 300, B).astype(np.int32)
        lens = np.where(pos >= 0, (pos + 1) // ratio, 0).astype(np.int32)
        stride = int(lens.max()) + 1
        rows = [rng.standard_normal(stride).astype(np.float32).tolist() for _ in range(B)]
        offs = rng.integers(0, 1000, B).astype(np.int32)
        swa = rng.integers(0, 100000, B).astype(np.int32)
        w = wl.custom("ragged", k, rows, out_offsets=offs.tolist())
        w["seq_lens"] = torch.from_numpy(lens)
        out, raw, _ = oracle.run_workload(w, mutant=mutant)
        width = k + window + 3
        res = oracle.swa_combine(out, raw, pos, window, swa, width, mutant=mutant)
        for b in range(B):
            topk_len = min(int(pos[b] + 1) // ratio, k) if pos[b] >= 0 else 0
            assert sorted(res[b, :topk_len].tolist()) == sorted(out[b, :topk_len].tolist())
            win = [t + int(swa[b]) for t in range(0, int(pos[b]) + 1) if int(pos[b]) - t < window]
            assert res[b, topk_len:topk_len + len(win)].tolist() == win
            assert (res[b, topk_len + len(win):] == -1).all()


PINS += [pin_swa_golden, pin_swa_formula]


LOGITS_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "indexer_logits_examples.json")


def pin_e4m3_codes(mutant=0):
    """Every FP8 E4M3 code decodes to torch's float8_e4m3fn value (a library
    routine for the same format); 0x7F and 0xFF are NaN."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if c in (0x7F, 0xFF):
            assert np.isnan(v) and np.isnan(lib[c])
        else:
            assert v == lib[c], (hex(c), v, lib[c])


def pin_logits_golden(mutant=0):
    """The indexer logits' hand-worked example (tests/golden/)."""
    with open(LOGITS_GOLDEN) as f:
        g = json.load(f)
    n_q = len(g["q"])
    out = np.full((n_q, g["stride"]), g["fill"], dtype=np.float32)
    oracle.indexer_logits(np.array(g["q"], dtype=np.uint8), np.array(g["kv"], dtype=np.uint8), g["kv_scale"],
                          g["weights"], g["ks"], g["ke"], out, mutant=mutant)
    assert out.tolist() == g["expect"]


def pin_logits_one_hot(mutant=0, seed=13):
    """Closed form at the indexer's own shape (64 heads of width 128): with
    q[t][h] one-hot at coordinate (h + t) % 128 and kv[s] one-hot at s % 128,
    only head h* = (s - t) mod 128 meets key s, so logits[t][s] = kv_scale[s]
    * w[t][h*] * max(0, q_val * kv_val) when h* < 64, else 0; windows clamp
    to [0, n_kv) and nothing outside them is written."""
    rng = np.random.default_rng(seed)
    n_q, heads, dim, n_kv = 6, 64, 128, 300
    f8 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    qc = rng.choice(finite, (n_q, heads))
    kc = rng.choice(finite, n_kv)
    q = np.zeros((n_q, heads, dim), np.uint8)
    kv = np.zeros((n_kv, dim), np.uint8)
    for t in range(n_q):
        for h in range(heads):
            q[t, h, (h + t) % dim] = qc[t, h]
    for s in range(n_kv):
        kv[s, s % dim] = kc[s]
    w = rng.standard_normal((n_q, heads)).astype(np.float32)
    scale = rng.uniform(0.25, 4.0, n_kv).astype(np.float32)
    ks = np.array([0, 5, -7, 150, 299, 200], np.int32)
    ke = np.array([300, 131, 40, 420, 299, 100], np.int32)
    out = np.full((n_q, n_kv + 3), -5.0, np.float32)
    oracle.indexer_logits(q, kv, scale, w, ks, ke, out, mutant=mutant)
    for t in range(n_q):
        lo, hi = max(int(ks[t]), 0), min(int(ke[t]), n_kv)
        for s in range(n_kv + 3):
            if not lo <= s < hi:
                assert out[t, s] == -5.0
                continue
            h = (s - t) % dim
            want = 0.0
            if h < heads:
                want = np.float64(scale[s]) * (np.float64(w[t, h]) * max(f8[qc[t, h]] * f8[kc[s]], 0.0))
            assert out[t, s] == np.float32(want), (t, s)


def pin_logits_invariants(mutant=0, seed=17):
    """What the definition fixes exactly, on random FP8 inputs: doubling the
    head weights or the key scales doubles every logit; negating every query
    code makes every head's dot product change sign, so w * max(0, -d) sums
    to what the original ReLU clipped (checked: the two runs' logits add up
    to kv_scale * sum_h w_h * |d_h|, computed here from |q . kv| by numpy);
    a common permutation of the heads (queries and weights) changes nothing
    beyond rounding."""
    rng = np.random.default_rng(seed)
    n_q, heads, dim, n_kv = 3, 8, 16, 40
    f8 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    q = rng.choice(finite, (n_q, heads, dim)).astype(np.uint8)
    kv = rng.choice(finite, (n_kv, dim)).astype(np.uint8)
    w = rng.standard_normal((n_q, heads)).astype(np.float32)
    scale = rng.uniform(0.5, 2.0, n_kv).astype(np.float32)
    ks, ke = np.zeros(n_q, np.int32), np.full(n_q, n_kv, np.int32)

    def run(q_, w_, s_):
        out = np.zeros((n_q, n_kv), np.float32)
        return oracle.indexer_logits(q_, kv, s_, w_, ks, ke, out, mutant=mutant).astype(np.float64)

    base = run(q, w, scale)
    assert np.array_equal(run(q, 2 * w, scale), 2 * base)
    assert np.array_equal(run(q, w, 2 * scale), 2 * base)
    neg = run(q ^ np.uint8(0x80), w, scale)  # the sign bit of every code flipped
    dots = np.einsum("thd,sd->ths", f8[q], f8[kv])
    absum = np.einsum("th,ths->ts", w.astype(np.float64), np.abs(dots)) * scale.astype(np.float64)
    assert np.allclose(base + neg, absum, rtol=1e-6, atol=1e-6 * np.abs(absum).max())
    perm = rng.permutation(heads)
    assert np.allclose(run(q[:, perm], w[:, perm], scale), base, rtol=1e-6, atol=1e-30)


PINS += [pin_e4m3_codes, pin_logits_golden, pin_logits_one_hot, pin_logits_invariants]


# ------------------------------------------------------------------ tests

@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()


def test_error_rows_are_empty_and_counted():
    w = wl.custom("ragged", 2, [[1.0, 2.0, 3.0], [4.0, 5.0, 6.0], [7.0, 8.0, 9.0]],
                  out_offsets=[0, 10, 20])
    w["seq_lens"] = torch.tensor([3, -1, 3], dtype=torch.int32)
    w["row_starts"] = torch.tensor([0, 0, -4], dtype=torch.int32)
    out, raw, err = oracle.run_workload(w)
    assert err == 2
    assert out[1].tolist() == [-1, -1] and out[2].tolist() == [-1, -1]
    assert sorted(out[0].tolist()) == [1, 2]


def test_planted_mistakes_are_caught():
    """Each planted mistake in the oracle fails at least one pin family."""
    for mutant in range(1, 13):
        caught = []
        for pin in PINS:
            try:
                pin(mutant=mutant)
            except AssertionError:
                caught.append(pin.__name__)
        assert caught, f"mutant {mutant} passed every pin"
