"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Small cases are compared element by element on every row; the full-size
workloads, in the launch configuration the benchmark times, are compared on
sampled rows. Deterministic mode must match the oracle bit-exactly (rows
sorted); default mode must select the bit-identical score multiset and pass
every invariant. No floating-point tolerance applies: selection does no
arithmetic on scores.
"""

from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_top_row_gb300 import workloads as wl
from topk_checks import HostWorkload, check_row_invariants, compare_with_oracle

pytestmark = pytest.mark.gpu

DET = 1
CANARY = 0x7EADBEEF


def assert_windows_in_bounds(w):
    """The library's contract: every row's 16-byte-aligned window span lies
    inside the score buffer (checked here so no test input reads past it)."""
    hw = HostWorkload(w)
    n = hw.scores.size
    for b in range(hw.batch):
        L = int(hw.seq_lens[b])
        s = hw.start(b)
        if L <= 0 or s < 0:
            continue
        rem = s % 4
        lo = b * hw.stride + s - rem
        hi = lo + 4 * ((L + rem + 3) // 4)
        assert 0 <= lo and hi <= n, f"row {b}: window [{lo}, {hi}) outside the {n}-element buffer"
        if hw.mode == "paged":
            t = b if hw.row_to_batch is None else int(hw.row_to_batch[b])
            t0 = 0 if hw.pt_row_starts is None else max(int(hw.pt_row_starts[b]), 0)
            need = (t0 + L + hw.page_size - 1) // hw.page_size
            assert need <= hw.pt_stride or hw.row_to_batch is None, f"row {b}: page-table row too short"
            assert t * hw.pt_stride + need <= hw.page_table.size, f"row {b}: page table too short"


def run_gpu(topk, w, flags, raw=True):
    assert_windows_in_bounds(w)
    w = wl.to_device(w, "cuda")
    B, k = int(w["batch"]), int(w["k"])
    out = torch.full((B, k), CANARY, dtype=torch.int32, device="cuda")
    out_raw = torch.full((B, k), CANARY, dtype=torch.int32, device="cuda") if raw else None
    before = w["scores"].clone()
    _, _, ws = topk.run_workload(w, out=out, out_raw=out_raw, flags=flags)
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int32), w["scores"].view(torch.int32)), "scores were written"
    o = out.cpu().numpy()
    r = out_raw.cpu().numpy() if raw else None
    assert not np.any(o == CANARY), "an output slot was not written"
    if raw:
        assert not np.any(r == CANARY), "an out_raw slot was not written"
    return o, r, ws


def check_full(topk, w, flags_list=(DET, 0)):
    hw = HostWorkload(w)
    ref_out, ref_raw, ref_err = oracle.run_workload_threads(w)
    for flags in flags_list:
        o, r, ws = run_gpu(topk, w, flags)
        compare_with_oracle(hw, o, r, ref_out, ref_raw, deterministic=bool(flags & DET))
        errs, dflags = topk.topk_read_device_errors(ws)
        assert errs == ref_err
        assert dflags == 0


# ---------------------------------------------------------------- golden examples

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def test_golden_examples(cuda_lib):
    from test_oracle_pins import _golden_workload
    for case in json.load(open(GOLDEN))["cases"]:
        w = _golden_workload(case)
        for flags in (DET, 0):
            o, r, _ = run_gpu(cuda_lib, w, flags)
            got = np.sort(o, axis=1).tolist()
            if flags & DET:
                assert got == case["det"], case["name"]
                assert np.sort(r, axis=1).tolist() == case["det_raw"], case["name"]
            else:
                assert got == case["det"] or got in case["also_valid"], case["name"]


# ---------------------------------------------------------------- small workloads, every row

SMALL = {
    "ragged_tiny": lambda: wl.ragged_tiny("cpu", sub_id=0),
    "ragged_tiny_s1": lambda: wl.ragged_tiny("cpu", sub_id=1),
    "paged_decode_small": lambda: wl.paged_decode("cpu", batch=16, seq_len=8192, k=2048),
    "paged_decode_k512": lambda: wl.paged_decode("cpu", batch=24, seq_len=4096, k=512, page_size=16),
    "ragged_extend_small": lambda: wl.ragged_extend("cpu", chunk=1, rows_per_chunk=40, n_req=2,
                                                    prefix=20000, new=40, k=2048),
    "paged_long_small": lambda: wl.paged_long("cpu", batch=2, seq_len=40000, k=2048),
    "paged_long_rows70": lambda: wl.paged_long("cpu", sub_id=3, batch=70, seq_len=20000, k=1024),
    "mixed_paged": lambda: wl.mixed("cpu", mode="paged", k=1024, batch=31, max_len=70000),
    "mixed_ragged": lambda: wl.mixed("cpu", mode="ragged", k=512, batch=31, max_len=70000),
    "mixed_ragged_b129": lambda: wl.mixed("cpu", mode="ragged", k=2048, batch=129, max_len=20000,
                                          sub_id=2),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_workload_every_row(cuda_lib, name):
    check_full(cuda_lib, SMALL[name]())


# ---------------------------------------------------------------- edge cases

def _rows(rng, lens, kind="normal"):
    rows = []
    for L in lens:
        if kind == "normal":
            rows.append(rng.standard_normal(L).astype(np.float32).tolist())
        elif kind == "ties":
            rows.append(rng.choice([-1.0, 0.0, 0.5, 1.0], size=L).astype(np.float32).tolist())
        elif kind == "equal":
            rows.append([0.25] * L)
        elif kind == "ascending":
            rows.append(np.linspace(-3, 3, L, dtype=np.float32).tolist())
        elif kind == "descending":
            rows.append(np.linspace(3, -3, L, dtype=np.float32).tolist())
        elif kind == "spread":  # each value alone in its 12-bit level-1 bin (up to 3200 distinct)
            code = np.resize(rng.permutation(3200), L)
            sign = np.where(code // 1600 == 1, -1.0, 1.0)
            e = (code % 1600) // 8 - 100
            m = code % 8
            rows.append((sign * np.ldexp(1.0 + m / 8.0, e)).astype(np.float32).tolist())
        elif kind == "narrow":  # one 14-bit prefix for every score, spread below it: the 12-bit levels' small-tie finish
            rows.append((1.0 + rng.random(L) / 64.0).astype(np.float32).tolist())
        elif kind == "negative":  # every score below zero: negative thresholds and bounds
            rows.append((-1.0 - np.abs(rng.standard_normal(L))).astype(np.float32).tolist())
        elif kind == "bf16":  # N(0, 0.01) rounded to bf16: long runs of equal keys at the threshold
            v = (rng.standard_normal(L) * 0.1).astype(np.float32)
            rows.append((v.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).tolist())
        elif kind == "special":
            v = rng.standard_normal(L).astype(np.float32)
            idx = rng.integers(0, L, size=max(1, L // 50))
            v[idx] = rng.choice(np.array([np.inf, -np.inf, -0.0, 0.0, np.finfo(np.float32).max,
                                          -np.finfo(np.float32).max], dtype=np.float32), size=idx.size)
            rows.append(v.tolist())
    return rows


@pytest.mark.parametrize("k", [1, 7, 512, 1000, 2048])
@pytest.mark.parametrize("mode", ["ragged", "paged"])
def test_boundary_lengths(cuda_lib, k, mode):
    rng = np.random.default_rng(k)
    lens = [0, 1, k - 1, k, k + 1, 8189, 8192, 8193, 16384, 16385, 40000]
    lens = [L for L in lens if L >= 0]
    starts = [int(x) for x in rng.integers(0, 4, size=len(lens))]
    w = wl.custom(mode, k, _rows(rng, lens), row_starts=starts,
                  out_offsets=[int(x) for x in rng.integers(0, 1 << 20, size=len(lens))],
                  page_size=64, seed=k)
    check_full(cuda_lib, w)


@pytest.mark.parametrize("kind", ["ties", "equal", "ascending", "descending", "special", "spread", "bf16",
                                  "negative", "narrow"])
@pytest.mark.parametrize("L", [3000, 8000, 12000, 50000])
def test_adversarial_values(cuda_lib, kind, L):
    """Heavy ties, one value everywhere, sorted rows (the first-tile estimate is
    then wrong or the candidate buffer overflows: the exact fallbacks run),
    infinities, signed zeros and the largest finite values; one value per
    level-1 bin (level 1 is exact); bf16-rounded values (equal keys beyond
    the second level); all-negative rows (negative thresholds and bounds);
    scores sharing one 14-bit key prefix (the register route falls back to
    its 12-bit levels and finishes there).
    L = 8000 puts a one-value row on the register route's fallback that
    keeps the levels in registers."""
    rng = np.random.default_rng(L)
    w = wl.custom("ragged", 2048, _rows(rng, [L, L // 2 + 1], kind), row_starts=[1, 2],
                  out_offsets=[0, 5])
    check_full(cuda_lib, w)


def test_cluster_path_with_adversarial_rows(cuda_lib):
    """Few long rows (cluster path): sorted, equal and tied values."""
    rng = np.random.default_rng(7)
    rows = _rows(rng, [70000], "ascending") + _rows(rng, [70001], "descending") + \
        _rows(rng, [65537], "equal") + _rows(rng, [100000], "ties")
    w = wl.custom("paged", 2048, rows, page_size=64, seed=7)
    check_full(cuda_lib, w)


@pytest.mark.parametrize("kind", ["bf16", "negative", "spread", "special"])
def test_cluster_path_value_kinds(cuda_lib, kind):
    """Cluster rows (B <= 64, L > 32768) on value kinds that steer the
    radix descent: bf16-rounded scores end the key descent early, negative
    scores give negative bounds, one value per level-1 bin makes level 1
    exact, and infinities/signed zeros/extreme finite values."""
    rng = np.random.default_rng(11)
    rows = _rows(rng, [40000, 131072, 65537], kind)
    w = wl.custom("ragged", 2048, rows, row_starts=[3, 1, 2], out_offsets=[0, 7, 1 << 20], seed=11)
    check_full(cuda_lib, w)


@pytest.mark.parametrize("k", [1, 33, 2048])
def test_small_tie_lists(cuda_lib, k):
    """Rows whose threshold value repeats a few times (up to 32 members: the
    one-warp ranking) and many times (the segmented ranking), on the register
    and streaming routes."""
    rng = np.random.default_rng(k)
    rows = []
    for L, reps in ((5000, 5), (5000, 40), (20000, 20), (20000, 300)):
        v = rng.standard_normal(L).astype(np.float32)
        order = np.sort(v)[::-1]
        thr = order[min(k, L) - 1]
        idx = rng.choice(L, size=reps, replace=False)
        v[idx] = thr  # the k-th largest value now occurs reps (+1) times
        rows.append(v.tolist())
    w = wl.custom("paged", k, rows, page_size=16, seed=k)
    check_full(cuda_lib, w)


@pytest.mark.parametrize("window,page_size", [(6000, 64), (16384, 16), (40000, 64), (20000, 1)])
def test_packed_paged_rows(cuda_lib, window, page_size):
    """Packed PAGED rows (topk_transform_paged_packed): batch-global score
    windows, request-local page-table starts, shared request tables; windows
    that put rows on the register, streaming and cluster routes."""
    w = wl.paged_packed("cpu", sub_id=window + page_size, n_req=3, q_rows=4, min_tokens=window // 2,
                        max_tokens=window + 9000, window=window, k=2048, page_size=page_size)
    check_full(cuda_lib, w)


def test_packed_paged_without_arrays_is_plain_paged(cuda_lib):
    """With neither packed array the packed entry point is the PAGED one."""
    w = wl.paged_decode("cpu", batch=6, seq_len=9000, k=700)
    d = wl.to_device(w, "cuda")
    ws = cuda_lib.new_workspace(6)
    cuda_lib.topk_plan(d["seq_lens"], 700, ws)
    a = torch.empty((6, 700), dtype=torch.int32, device="cuda")
    b = torch.empty_like(a)
    cuda_lib.topk_transform_paged(d["scores"], d["score_stride"], None, d["seq_lens"], d["page_table"],
                                  d["page_table_stride"], d["page_size"], 700, ws, a, flags=DET)
    cuda_lib.topk_transform_paged_packed(d["scores"], d["score_stride"], None, d["seq_lens"], d["page_table"],
                                         d["page_table_stride"], d["page_size"], None, None, 700, ws, b, flags=DET)
    torch.cuda.synchronize()
    assert torch.equal(torch.sort(a, dim=1).values, torch.sort(b, dim=1).values)


@pytest.mark.parametrize("mode", ["paged", "ragged"])
def test_cluster_floor_lengths(cuda_lib, mode):
    """Rows either side of the cluster floor (32768) in a small batch: 32768
    stays on the streaming route, 32769 and longer take the cluster route."""
    rng = np.random.default_rng(32768)
    lens = [32767, 32768, 32769, 32772, 36000]
    starts = [int(x) for x in rng.integers(0, 4, size=len(lens))]
    w = wl.custom(mode, 2048, _rows(rng, lens), row_starts=starts,
                  out_offsets=[int(x) for x in rng.integers(0, 1 << 20, size=len(lens))], page_size=64, seed=5)
    check_full(cuda_lib, w)


@pytest.mark.parametrize("batch", [39, 64, 65])
def test_cluster_batch_limits(cuda_lib, batch):
    """Mixed lengths up to 70000 around the cluster path's batch limits: up to
    64 rows the long rows take the cluster kernel (its two-CTA-per-SM build
    once the rows outnumber the clusters that fit one CTA per SM, 36 on a
    GB300), at 65 they stay on the streaming route."""
    w = wl.mixed("cpu", mode="paged", k=1024, batch=batch, max_len=70000, sub_id=batch)
    check_full(cuda_lib, w)


def test_largest_batch_in_one_launch(cuda_lib):
    """16384 rows (the largest batch of the pages' workloads) in one plan and
    one transform: short RAGGED rows at unaligned starts, k=256."""
    w = wl.mixed("cpu", mode="ragged", k=256, batch=16384, max_len=3000, min_len=16, sub_id=16384)
    check_full(cuda_lib, w)


def test_packed_negative_table_start_is_a_data_error(cuda_lib):
    w = wl.paged_packed("cpu", sub_id=5, n_req=2, q_rows=3, min_tokens=3000, max_tokens=5000, window=4000,
                        k=512, page_size=64)
    w["page_table_row_starts"] = w["page_table_row_starts"].clone()
    w["page_table_row_starts"][2] = -1
    check_full(cuda_lib, w)


def test_nan_scores_order_deterministically(cuda_lib):
    rng = np.random.default_rng(11)
    v = rng.standard_normal(20000).astype(np.float32)
    v[rng.integers(0, 20000, 30)] = np.nan
    v[rng.integers(0, 20000, 30)] = -np.nan
    w = wl.custom("ragged", 100, [v.tolist()], out_offsets=[0])
    hw = HostWorkload(w)
    ref_out, ref_raw, _ = oracle.run_workload(w)
    o, r, _ = run_gpu(cuda_lib, w, DET)
    np.testing.assert_array_equal(np.sort(r), np.sort(ref_raw))


def test_no_row_starts_and_no_out_raw(cuda_lib):
    w = wl.paged_decode("cpu", batch=4, seq_len=10000, k=300, page_size=8)
    hw = HostWorkload(w)
    ref_out, _, _ = oracle.run_workload(w)
    o, r, _ = run_gpu(cuda_lib, w, DET, raw=False)
    np.testing.assert_array_equal(np.sort(o, axis=1), np.sort(ref_out, axis=1))


@pytest.mark.parametrize("route", ["trivial", "register", "streaming", "cluster", "streaming_many"])
@pytest.mark.parametrize("mode", ["paged", "ragged"])
def test_without_out_raw_on_every_route(cuda_lib, route, mode):
    """out_raw = NULL on each route (trivial L <= k; register L <= 8192;
    streaming longer rows; cluster rows: L > 32768 in a batch of at most 64;
    streaming_many: the same long rows in a batch of 65, off the cluster
    path): the outputs alone match the oracle."""
    rng = np.random.default_rng(len(route) + (7 if mode == "paged" else 0))
    lens = {"trivial": [1, 300, 512], "register": [513, 4000, 8192], "streaming": [8193, 20000, 32768],
            "cluster": [32769, 70000, 131072], "streaming_many": [40000] * 65}[route]
    starts = [int(x) for x in rng.integers(0, 4, size=len(lens))]
    w = wl.custom(mode, 512, _rows(rng, lens), row_starts=starts,
                  out_offsets=[int(x) for x in rng.integers(0, 1 << 20, size=len(lens))], page_size=16,
                  seed=len(lens))
    ref_out, _, _ = oracle.run_workload_threads(w)
    for flags in (DET, 0):
        o, _, _ = run_gpu(cuda_lib, w, flags, raw=False)
        if flags & DET:
            np.testing.assert_array_equal(np.sort(o, axis=1), np.sort(ref_out, axis=1))
        else:  # equal scores may swap: the positions behind the outputs select the same scores
            hw = HostWorkload(w)
            for b in range(hw.batch):
                L = hw.length(b)
                slots = hw.transform(b, np.arange(L))           # position -> output value
                pos_of = {int(v): p for p, v in enumerate(slots)}
                got = [pos_of[int(v)] for v in o[b] if v >= 0]
                ref = [pos_of[int(v)] for v in ref_out[b] if v >= 0]
                win = hw.window(b)
                assert len(got) == len(set(got)) == len(ref), f"row {b}"
                np.testing.assert_array_equal(np.sort(win[got].view(np.uint32)), np.sort(win[ref].view(np.uint32)))


@pytest.mark.parametrize("page_size", [1, 2, 4096, 1 << 19])
def test_page_sizes(cuda_lib, page_size):
    rng = np.random.default_rng(page_size)
    L = 9000
    pages = (L + page_size - 1) // page_size
    table = rng.permutation(3 * pages).reshape(3, pages) if page_size < 4096 else \
        rng.integers(0, 1 << 31 >> 19, size=(3, pages))
    w = wl.custom("paged", 777, _rows(rng, [L, L, 5000]), page_size=page_size,
                  page_table=table.astype(np.int32))
    check_full(cuda_lib, w)


def test_shared_buffer_stride_zero(cuda_lib):
    w = wl.ragged_tiny("cpu", sub_id=5, batch=40, k=100, max_len=20000)
    check_full(cuda_lib, w)


def test_data_errors_are_counted(cuda_lib):
    rng = np.random.default_rng(3)
    w = wl.custom("ragged", 16, _rows(rng, [100, 100, 100, 100]), out_offsets=[0, 0, 0, 0])
    w["seq_lens"] = torch.tensor([100, -5, 100, 100], dtype=torch.int32)
    w["row_starts"] = torch.tensor([0, 0, -8, 0], dtype=torch.int32)
    ref_out, ref_raw, ref_err = oracle.run_workload(w)
    assert ref_err == 2
    o, r, ws = run_gpu(cuda_lib, w, DET)
    np.testing.assert_array_equal(np.sort(o, axis=1), np.sort(ref_out, axis=1))
    errs, flags = cuda_lib.topk_read_device_errors(ws)
    assert errs == 2 and flags == 0


def test_plan_mismatch_still_exact(cuda_lib):
    """A transform whose (batch, k) differs from the plan's flags it and still
    computes every row exactly (without the cluster path)."""
    w = wl.to_device(wl.paged_long("cpu", batch=3, seq_len=70000, k=512), "cuda")
    ref_out, ref_raw, _ = oracle.run_workload(w)
    ws = cuda_lib.new_workspace(3)
    cuda_lib.topk_plan(w["seq_lens"], 256, ws)  # planned for another k
    out = torch.full((3, 512), CANARY, dtype=torch.int32, device="cuda")
    raw = torch.full((3, 512), CANARY, dtype=torch.int32, device="cuda")
    cuda_lib.topk_transform_paged(w["scores"], w["score_stride"], None, w["seq_lens"], w["page_table"],
                                  w["page_table_stride"], 64, 512, ws, out, raw, DET)
    np.testing.assert_array_equal(np.sort(raw.cpu().numpy(), 1), np.sort(ref_raw, 1))
    errs, flags = cuda_lib.topk_read_device_errors(ws)
    assert flags & cuda_lib.TOPK_DEVICE_FLAG_PLAN_MISMATCH


def test_one_plan_serves_many_transforms(cuda_lib):
    w = wl.to_device(wl.mixed("cpu", mode="ragged", k=512, batch=20, max_len=50000, sub_id=9), "cuda")
    ref_out, ref_raw, _ = oracle.run_workload(w)
    ws = cuda_lib.new_workspace(20)
    cuda_lib.topk_plan(w["seq_lens"], 512, ws)
    for _ in range(3):
        out, _, _ = cuda_lib.run_workload(w, workspace=ws, flags=DET, plan=False)
        np.testing.assert_array_equal(np.sort(out.cpu().numpy(), 1), np.sort(ref_out, 1))


def test_deterministic_mode_is_repeatable(cuda_lib):
    w = wl.to_device(wl.paged_long("cpu", batch=31, seq_len=50000, k=2048, sub_id=1), "cuda")
    outs = [np.sort(cuda_lib.run_workload(w, flags=DET)[0].cpu().numpy(), 1) for _ in range(3)]
    assert all(np.array_equal(outs[0], x) for x in outs[1:])


def test_non_default_stream(cuda_lib):
    w = wl.to_device(wl.paged_decode("cpu", batch=8, seq_len=8192, k=2048), "cuda")
    ref_out, _, _ = oracle.run_workload(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, _, _ = cuda_lib.run_workload(w, flags=DET, stream=s)
    s.synchronize()
    np.testing.assert_array_equal(np.sort(out.cpu().numpy(), 1), np.sort(ref_out, 1))


# ---------------------------------------------------------------- full sizes, every row

def _check_every_row(topk, w_dev, flags=(DET, 0)):
    """The whole launch, as the benchmark times it (one plan + one transform
    over every row), against the oracle on every row."""
    assert_windows_in_bounds(w_dev)
    w_host = wl.to_device(w_dev, "cpu")
    hw = HostWorkload(w_host)
    ref_out, ref_raw, ref_err = oracle.run_workload_threads(w_host)
    B, k = int(w_dev["batch"]), int(w_dev["k"])
    for f in flags:
        out = torch.full((B, k), CANARY, dtype=torch.int32, device="cuda")
        raw = torch.full((B, k), CANARY, dtype=torch.int32, device="cuda")
        _, _, ws = topk.run_workload(w_dev, out=out, out_raw=raw, flags=f)
        torch.cuda.synchronize()
        o, r = out.cpu().numpy(), raw.cpu().numpy()
        assert not np.any(o == CANARY) and not np.any(r == CANARY)
        compare_with_oracle(hw, o, r, ref_out, ref_raw, deterministic=bool(f & DET))
        assert topk.topk_read_device_errors(ws) == (ref_err, 0)


@pytest.mark.slow
@pytest.mark.parametrize("chunk", [0, 9])
def test_full_ragged_extend_chunk_every_row(cuda_lib, chunk):
    """A full 1024-row chunk of the prefill-extend workload (rows of
    28673..32768 scores at stride 131072): every row, both modes."""
    _check_every_row(cuda_lib, wl.ragged_extend("cuda", chunk=chunk))


@pytest.mark.slow
@pytest.mark.parametrize("mode", ["paged", "ragged"])
def test_full_mixed_b1024_k2048_every_row(cuda_lib, mode):
    """The mixed sweep's largest launch (1024 rows, log-uniform lengths up to
    131072 plus the boundary rows, k = 2048): every row, both modes."""
    _check_every_row(cuda_lib, wl.mixed("cuda", mode=mode, k=2048, batch=1024, sub_id=1024))


# ---------------------------------------------------------------- full sizes, sampled rows

def _sample_and_check(topk, w, rows, flags=(DET, 0)):
    assert_windows_in_bounds(w)
    hw_rows = wl.select_rows(w, rows)
    ref_out, ref_raw, _ = oracle.run_workload(hw_rows)
    hw = HostWorkload(hw_rows)
    for f in flags:
        B, k = int(w["batch"]), int(w["k"])
        out = torch.full((B, k), CANARY, dtype=torch.int32, device="cuda")
        raw = torch.full((B, k), CANARY, dtype=torch.int32, device="cuda")
        topk.run_workload(w, out=out, out_raw=raw, flags=f)
        idx = torch.tensor(rows, device="cuda")
        o = out[idx].cpu().numpy()
        r = raw[idx].cpu().numpy()
        compare_with_oracle(hw, o, r, ref_out, ref_raw, deterministic=bool(f & DET))
        # every row: count and padding invariants on the device copy
        valid = (raw >= 0).sum(1)
        lens = w["seq_lens"].clamp(min=0).clamp(max=k)
        assert torch.equal(valid.to(torch.int32), lens.to(torch.int32))
        assert not bool((out == CANARY).any())


@pytest.mark.slow
def test_full_paged_decode(cuda_lib):
    w = wl.paged_decode("cuda")
    _sample_and_check(cuda_lib, w, [0, 1, 63, 127])


@pytest.mark.slow
@pytest.mark.parametrize("chunk", [0, 7, 15])
def test_full_ragged_extend_chunk(cuda_lib, chunk):
    w = wl.ragged_extend("cuda", chunk=chunk)
    _sample_and_check(cuda_lib, w, [0, 1, 511, 1023])


@pytest.mark.slow
@pytest.mark.parametrize("batch", [1, 30, 31])
def test_full_paged_long(cuda_lib, batch):
    w = wl.paged_long("cuda", batch=batch, sub_id=batch)
    _sample_and_check(cuda_lib, w, sorted({0, batch // 2, batch - 1}))


@pytest.mark.slow
@pytest.mark.parametrize("mode", ["paged", "ragged"])
@pytest.mark.parametrize("k", [512, 1024, 2048])
@pytest.mark.parametrize("batch", [1, 31, 129, 1024])
def test_full_mixed_sweep(cuda_lib, mode, k, batch):
    w = wl.mixed("cuda", mode=mode, k=k, batch=batch, sub_id=batch)
    rows = sorted(set(range(min(batch, 9))) | {batch // 2, batch - 1})
    _sample_and_check(cuda_lib, w, rows)


@pytest.mark.slow
@pytest.mark.parametrize("bi", range(9))
def test_full_mixed_boundary_single_rows(cuda_lib, bi):
    for mode in ("paged", "ragged"):
        w = wl.mixed("cuda", mode=mode, k=2048, batch=1, boundary_index=bi, sub_id=50 + bi)
        _sample_and_check(cuda_lib, w, [0])


@pytest.mark.slow
@pytest.mark.parametrize("name", ["extend", "decode"])
def test_fast_path_takes_every_row(cuda_lib, name):
    """The sample bounds hold on the benchmark's workloads: no row of a full
    extend chunk (256-thread rows kernel, spread sample) or of the decode batch
    (512-thread rows kernel, register sample) falls back to the exact path,
    going by the plan header's count of exact-path rows."""
    w = wl.ragged_extend("cuda", chunk=3) if name == "extend" else wl.paged_decode("cuda")
    _, _, ws = cuda_lib.run_workload(w)
    torch.cuda.synchronize()
    hdr = ws[:64].cpu().numpy().view(np.uint32)
    assert hdr[7] == 0, f"{hdr[7]} rows took the exact path"


# ---------------------------------------------------------------- the fused SWA combine

def _check_swa(topk, w, flags_list=(DET, 0)):
    """topk_transform_ragged_swa against the oracle's transform + combine: the
    window tail of every row bit-exact, the top-k part as the plain transform
    is checked (sets in deterministic mode, score multisets otherwise)."""
    assert_windows_in_bounds(w)
    hw = HostWorkload(w)
    ref_out, ref_raw, ref_err = oracle.run_workload(w)
    width, k, B = int(w["out_width"]), int(w["k"]), int(w["batch"])
    offs = None if w.get("swa_offsets") is None else w["swa_offsets"].cpu().numpy()
    ref = oracle.swa_combine(ref_out, ref_raw, w["positions"].cpu().numpy(), int(w["window_size"]), offs, width)
    topk_len = np.array([min(hw.length(b), k) for b in range(B)])
    d = wl.to_device(w, "cuda")
    for flags in flags_list:
        out = torch.full((B, width), CANARY, dtype=torch.int32, device="cuda")
        raw = torch.full((B, k), CANARY, dtype=torch.int32, device="cuda")
        _, _, ws = topk.run_workload(d, out=out, out_raw=raw, flags=flags)
        torch.cuda.synchronize()
        o, r = out.cpu().numpy(), raw.cpu().numpy()
        assert not np.any(o == CANARY) and not np.any(r == CANARY)
        gpu_topk = np.full((B, k), -1, dtype=np.int32)
        for b in range(B):
            n = int(topk_len[b])
            assert o[b, n:].tolist() == ref[b, n:].tolist(), f"row {b}: window tail"
            gpu_topk[b, :n] = o[b, :n]
        compare_with_oracle(hw, gpu_topk, r, ref_out, ref_raw, deterministic=bool(flags & DET))
        assert topk.topk_read_device_errors(ws) == (ref_err, 0)


@pytest.mark.parametrize("route,kw", [
    ("register_512", dict(n_req=2, new=48)),                      # 96 rows, L ~ 7168: 512-thread register route
    ("streaming_256", dict(n_req=2, new=100)),                    # 200 rows (> SMs): 256-thread streaming route
    ("cluster", dict(n_req=2, new=6, prefix=40000, ratio=1)),     # 12 rows of L ~ 40001: cluster route
    ("trivial", dict(n_req=1, new=300, prefix=0, ratio=128)),     # L <= 2 <= k, windows cut at token 0
    ("k2048", dict(n_req=3, new=70, k=2048, window=64)),          # 210 rows, k = 2048
])
def test_swa_combine_routes(cuda_lib, route, kw):
    _check_swa(cuda_lib, wl.ragged_swa("cpu", sub_id=len(route), **kw))


def test_swa_combine_edge_rows(cuda_lib):
    """Negative positions (no window), a data-error row, a window wider than
    the prefix, no SWA offsets, and an output wider than k + window."""
    rng = np.random.default_rng(5)
    rows = [rng.standard_normal(n).astype(np.float32).tolist() for n in (600, 3, 1, 40, 9000)]
    w = wl.custom("ragged", 32, rows, out_offsets=[7, 0, 5, 1000, 3])
    w["seq_lens"] = torch.tensor([600, 3, -1, 40, 9000], dtype=torch.int32)
    w.update(positions=torch.tensor([-1, 2, 10, 5000, 0], dtype=torch.int32), window_size=16,
             swa_offsets=None, out_width=52)
    _check_swa(cuda_lib, w)


@pytest.mark.slow
def test_row_beyond_the_compact_index(cuda_lib):
    """A row longer than the compact lists' 16-bit index covers on the
    256-thread build (4096 tiles of 4096 scores): it takes the per-warp
    region filter (two register tiles). 160 rows (more than the SMs) share one
    buffer (stride 0): one of 2^24 + 5000 scores, the others of 3000."""
    g = torch.Generator().manual_seed(77)
    L = (1 << 24) + 5000
    scores = torch.randn(L + 64, generator=g)
    B, k = 160, 2048
    lens = torch.full((B,), 3000, dtype=torch.int32)
    lens[0] = L
    w = dict(name="beyond the compact index", mode="ragged", k=k, scores=scores, score_stride=0,
             row_starts=torch.arange(B, dtype=torch.int32) * 3, seq_lens=lens,
             out_offsets=torch.arange(B, dtype=torch.int32), page_table=None, page_table_stride=0,
             page_size=1, batch=B)
    check_full(cuda_lib, w)


# ---------------------------------------------------------------- thresholds far above the sample bound

def _far_threshold_rows(batch, length, seed):
    """Rows whose k-th score lies many 16-bit prefix steps above the sample's
    bound: (a) scores in [1e-7, 1e-6) with 2300 (rows of 30000) or 2100
    (other lengths) in [0.5, 1) at random places, (b) N(-0.3 z, 0.3) with z
    the normal quantile of the k-th largest (k = 2048), so that it sits near
    0 and the bound falls among the negative scores, (c) N(0, 1) rows."""
    g = torch.Generator().manual_seed(seed)
    rows = []
    for b in range(batch):
        kind = b % 3
        if kind == 0:
            r = 1e-7 + 9e-7 * torch.rand(length, generator=g)
            n_big = {30000: 2300}.get(length, 2100)
            idx = torch.randperm(length, generator=g)[:n_big]
            r[idx] = 0.5 + 0.5 * torch.rand(n_big, generator=g)
        elif kind == 1:
            z = {60000: 1.82, 30000: 1.49, 8192: 0.67, 4096: 0.0}[length]  # the normal quantile of the k-th largest
            r = -z * 0.3 + 0.3 * torch.randn(length, generator=g)
        else:
            r = torch.randn(length, generator=g)
        rows.append(r)
    scores = torch.stack(rows).to(torch.float32).contiguous()
    B = batch
    return dict(mode="ragged", k=2048, scores=scores.reshape(-1), score_stride=length, row_starts=None,
                seq_lens=torch.full((B,), length, dtype=torch.int32),
                out_offsets=(torch.arange(B, dtype=torch.int32) * length).contiguous(), page_table=None,
                page_table_stride=0, page_size=1, batch=B, name=f"far thresholds B={B}")


def _paged_far_rows(batch, length, seed, page_size=64):
    """_far_threshold_rows in PAGED mode: each row's own random page table."""
    w = _far_threshold_rows(batch, length, seed)
    pages = (length + page_size - 1) // page_size
    g = torch.Generator().manual_seed(seed + 1)
    w.update(mode="paged", out_offsets=None, page_size=page_size, page_table_stride=pages,
             page_table=torch.randperm(batch * pages, generator=g).to(torch.int32).view(batch, pages).contiguous())
    return w


@pytest.mark.parametrize("mode", ["ragged", "paged"])
@pytest.mark.parametrize("batch,length,fast", [(200, 30000, True), (100, 30000, True), (100, 8192, True),
                                               (200, 4096, False), (20, 60000, True)])
def test_threshold_far_above_the_bound(cuda_lib, batch, length, fast, mode):
    """Rows whose threshold lies beyond the finish's first window of 255
    prefixes over the bound are finished by re-binning the top bin's members
    (no exact path: `fast`), and match the oracle: streamed rows on the
    compact lists (30000 scores: the 256-thread rows kernel for 200 rows, the
    512-thread one for 100), register rows on the 512-thread kernel (8192
    scores) and long rows on the cluster kernel (20 rows of 60000, four CTAs
    a row, the windows' histograms merged over the cluster); the 256-thread
    kernel's register rows (4096 scores) take the exact path instead."""
    seed = 31 + batch + length
    w = _far_threshold_rows(batch, length, seed) if mode == "ragged" else _paged_far_rows(batch, length, seed)
    hw = HostWorkload(w)
    ref_out, ref_raw, err = oracle.run_workload(w)
    assert err == 0
    d = wl.to_device(w, "cuda")
    for flags in (DET, 0):
        out = torch.full((batch, 2048), CANARY, dtype=torch.int32, device="cuda")
        out_raw = torch.full((batch, 2048), CANARY, dtype=torch.int32, device="cuda")
        _, _, ws = cuda_lib.run_workload(d, out=out, out_raw=out_raw, flags=flags)
        torch.cuda.synchronize()
        hdr = ws[:64].cpu().numpy().view(np.uint32)
        if fast:
            assert hdr[7] == 0, f"{hdr[7]} rows took the exact path"
        compare_with_oracle(hw, out.cpu().numpy(), out_raw.cpu().numpy(), ref_out, ref_raw,
                            deterministic=flags == DET)
