"""GPU parity of the indexer logits (the FP8 MQA-logits producer upstream of
the top-k) against the CPU oracle, through the C ABI.

The oracle's dot products are exact (fp64) and its head sum is fp64; the
kernel accumulates the 128 exact FP8 products of a dot product in fp32 on the
tensor cores, then sums the 64 weighted ReLUs in fp32. Its error is at most
about 150 fp32 roundings of the magnitude sum
M[t][s] = kv_scale[s] * sum_h |w[t][h]| * sum_d |q[t][h][d] * kv[s][d]|,
about 2^-17 * M; the tests allow 2^-12 * M (room for the tensor cores'
unspecified internal accumulation order), far below the O(M) error of any
mix-up of heads, keys, queries or weights. Columns outside a row's window
must keep the buffer's sentinel bit for bit. The top-k fed by the kernel's
logits is compared with the oracle's top-k of the same logits, exactly.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_top_row_gb300 import workloads as wl
from topk_checks import HostWorkload, compare_with_oracle

pytestmark = pytest.mark.gpu

FILL = -12345.0
REL_TOL = 2.0 ** -12


def e4m3_f64(codes):
    """FP8 E4M3 codes -> float64 (torch's float8_e4m3fn conversion)."""
    return torch.as_tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def host(w):
    return {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) else v) for k, v in w.items()}


def run_gpu(w, stride=None, rows=None):
    """The kernel on workload w (moved to the GPU); returns the float32 logits
    [n_q, stride] on the host, every column not written holding FILL."""
    topk = pytest.importorskip("sparse_attention_top_row_gb300")
    n_q, n_kv = w["n_q"], w["n_kv"]
    stride = stride or n_kv + 5
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    logits = torch.full((n_q, stride), FILL, dtype=torch.float32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    topk.topk_indexer_logits(d["q"], d["kv"], d["kv_scale"], d["weights"], d["ks"], d["ke"], logits, stride, flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0, "a bounded wait gave up"
    return logits if rows is None else logits[rows]


def oracle_rows(hw, rows, col_lo, col_hi, stride):
    """The oracle's logits of the given query rows over columns [col_lo,
    col_hi) of each (clipped to the row's window), FILL elsewhere."""
    n = len(rows)
    ks = np.maximum(hw["ks"][rows], col_lo)
    ke = np.minimum(hw["ke"][rows], col_hi)
    out = np.full((n, stride), FILL, np.float32)
    oracle.indexer_logits(hw["q"][rows], hw["kv"], hw["kv_scale"], hw["weights"][rows], ks, ke, out)
    return out


def magnitude(hw, rows, cols):
    """M[i][j] for query rows[i], key cols[j] (see the module docstring)."""
    aq = np.abs(e4m3_f64(hw["q"][rows]))                      # [n, H, D]
    akv = np.abs(e4m3_f64(hw["kv"][cols]))                    # [c, D]
    dots = aq @ akv.T                                         # [n, H, c]
    aw = np.abs(hw["weights"][rows].astype(np.float64))      # [n, H]
    return np.einsum("nh,nhc->nc", aw, dots) * hw["kv_scale"][cols].astype(np.float64)[None, :]


def check_rows(gpu, hw, rows, col_lo, col_hi):
    """GPU rows (host float32, full width) against the oracle on [col_lo, col_hi)."""
    stride = gpu.shape[1]
    col_lo, col_hi = max(col_lo, 0), min(col_hi, stride)
    want = oracle_rows(hw, rows, col_lo, col_hi, stride)
    cols = np.arange(col_lo, min(col_hi, hw["n_kv"]))
    for i, t in enumerate(rows):
        lo, hi = max(int(hw["ks"][t]), col_lo, 0), min(int(hw["ke"][t]), col_hi, hw["n_kv"])
        g, o = gpu[i], want[i]
        inside = np.zeros(stride, bool)
        if lo < hi:
            inside[lo:hi] = True
        span = slice(col_lo, col_hi)
        outside = ~inside[span]
        assert (g[span][outside] == FILL).all(), f"row {t}: a column outside the window was written"
        if lo >= hi:
            continue
        m = magnitude(hw, [t], np.arange(lo, hi))[0]
        err = np.abs(g[lo:hi].astype(np.float64) - o[lo:hi].astype(np.float64))
        bad = err > REL_TOL * m + 1e-30
        assert not bad.any(), (f"row {t}: {bad.sum()} columns off, worst at {lo + int(np.argmax(err - REL_TOL * m))}: "
                               f"max err/M = {float((err / np.maximum(m, 1e-30)).max()):.3g}")
    return cols


@pytest.mark.parametrize("n_q,n_kv,sub", [(1, 1, 0), (5, 127, 1), (13, 1000, 2), (8, 4096, 3), (21, 777, 4)])
def test_logits_random_windows(cuda_lib, n_q, n_kv, sub):
    """Every row, every column: random windows (empty, reversed, clamped at
    both ends, unaligned to the 128-key tiles), groups of 4 queries with a
    ragged last group."""
    w = wl.indexer_inputs("cpu", sub, n_q=n_q, n_kv=n_kv)
    hw = host(w)
    gpu = run_gpu(w).cpu().numpy()
    check_rows(gpu, hw, np.arange(n_q), 0, n_kv + 5)


def test_logits_window_edges(cuda_lib):
    """Hand-picked windows: one key, one whole tile, tile-straddling spans,
    an empty and a reversed window, the last key, a window past both ends."""
    n_kv = 1031
    windows = ([0, 127, 128, 100, 500, 500, 1030, -50, 3, 256, 900],
               [1, 128, 256, 300, 500, 400, 1031, 2000, 1030, 257, 1031])
    w = wl.indexer_inputs("cpu", 5, n_q=11, n_kv=n_kv, windows=windows)
    hw = host(w)
    gpu = run_gpu(w, stride=n_kv + 16).cpu().numpy()
    check_rows(gpu, hw, np.arange(11), 0, n_kv + 16)


def test_logits_special_values(cuda_lib):
    """Extreme codes: +-448 (the largest finite), the subnormals, signed
    zeros; every dot product of a query with a key made of the same byte."""
    n_q, n_kv = 4, 256
    codes = np.array([0x7E, 0xFE, 0x01, 0x81, 0x00, 0x80, 0x38, 0xB8], np.uint8)
    q = np.zeros((n_q, 64, 128), np.uint8)
    for t in range(n_q):
        for h in range(64):
            q[t, h] = codes[(t + h) % len(codes)]
    kv = np.array([codes[s % len(codes)] for s in range(n_kv)], np.uint8)[:, None].repeat(128, 1)
    rng = np.random.default_rng(7)
    w = dict(q=torch.from_numpy(q), kv=torch.from_numpy(np.ascontiguousarray(kv)),
             kv_scale=torch.from_numpy(rng.uniform(0.5, 2.0, n_kv).astype(np.float32)),
             weights=torch.from_numpy(rng.standard_normal((n_q, 64)).astype(np.float32)),
             ks=torch.zeros(n_q, dtype=torch.int32), ke=torch.full((n_q,), n_kv, dtype=torch.int32),
             n_q=n_q, n_kv=n_kv)
    hw = host(w)
    gpu = run_gpu(w).cpu().numpy()
    check_rows(gpu, hw, np.arange(n_q), 0, n_kv)


def test_logits_extend_chunk_sampled(cuda_lib):
    """The extend chunk the benchmark times (1024 queries over 131072 keys,
    windows of 28673..29696 keys): sampled rows, each at its window's head,
    tail and an interior span, plus the columns just outside the window."""
    w = wl.indexer_extend("cuda", 0)
    stride = w["stride"]
    gpu = run_gpu(w, stride=stride)
    hw = host(w)
    rows = [0, 1, 2, 3, 4, 511, 1022, 1023]
    sample = gpu[rows].cpu().numpy()
    del gpu
    for i, t in enumerate(rows):
        ks, ke = int(hw["ks"][t]), int(hw["ke"][t])
        for lo, hi in ((ks - 3, ks + 160), (ke - 160, ke + 3), (ks + 9000, ks + 9300)):
            check_rows(sample[i:i + 1], {**hw, "q": hw["q"][[t]], "weights": hw["weights"][[t]],
                                         "ks": hw["ks"][[t]], "ke": hw["ke"][[t]]}, np.array([0]), lo, hi)


def test_logits_feed_the_topk(cuda_lib):
    """The logits rows go straight into the RAGGED top-k (row_start = ks,
    seq_len = ke - ks, out_offsets = ks): the top-k of the kernel's logits
    equals the oracle's top-k of the same logits."""
    topk = cuda_lib
    n_q, n_kv, k = 24, 12000, 2048
    starts = np.array([0, 0, 100, 4000, 0, 7, 5000, 11000] * 3, np.int64)[:n_q]
    lens = np.array([12000, 2047, 2048, 2049, 8192, 9000, 7000, 1000] * 3, np.int64)[:n_q]
    w = wl.indexer_inputs("cuda", 6, n_q=n_q, n_kv=n_kv, windows=(starts, starts + lens))
    stride = n_kv + 4
    logits = run_gpu(w, stride=stride)
    tw = dict(mode="ragged", k=k, scores=logits.reshape(-1), score_stride=stride, row_starts=w["ks"],
              seq_lens=(w["ke"] - w["ks"]).to(torch.int32), out_offsets=w["ks"], page_table=None,
              page_table_stride=0, page_size=1, batch=n_q, name="indexer logits -> ragged top-k")
    hw = HostWorkload(tw)
    ref_out, ref_raw, err = oracle.run_workload(tw)
    assert err == 0
    for flags in (0, 1):
        out = torch.full((n_q, k), 0x7EADBEEF, dtype=torch.int32, device="cuda")
        out_raw = torch.full((n_q, k), 0x7EADBEEF, dtype=torch.int32, device="cuda")
        topk.run_workload(tw, out=out, out_raw=out_raw, flags=flags)
        torch.cuda.synchronize()
        compare_with_oracle(hw, out.cpu().numpy(), out_raw.cpu().numpy(), ref_out, ref_raw,
                            deterministic=flags == 1)


@pytest.mark.parametrize("n_q,n_kv,sub,rows", [
    (1000, 5000, 7, [0, 1, 2, 3, 4, 5, 250, 251, 500, 997, 998, 999]),  # 3 units a group, ~5 units a CTA
    (37, 20000, 8, [0, 1, 2, 35, 36]),                                   # 15 units a group, a partial last group
])
def test_logits_work_units(cuda_lib, n_q, n_kv, sub, rows):
    """The persistent kernel's work units: groups split into several key
    shares, CTAs walking several units (the query tiles and records double-
    buffered), empty units skipped, a partial last group; sampled rows, every
    column, against the oracle."""
    w = wl.indexer_inputs("cpu", sub, n_q=n_q, n_kv=n_kv)
    hw = host(w)
    gpu = run_gpu(w, rows=rows).cpu().numpy()
    sub_hw = {**hw, "q": hw["q"][rows], "weights": hw["weights"][rows], "ks": hw["ks"][rows], "ke": hw["ke"][rows]}
    check_rows(gpu, sub_hw, np.arange(len(rows)), 0, n_kv + 5)


def test_logits_chain_in_a_cuda_graph(cuda_lib):
    """The producer -> plan -> transform chain captured in a CUDA graph (the
    three launches with programmatic dependent launch, as a serving step runs
    them) and replayed on fresh inputs: the top-k of the replayed logits is the
    oracle's top-k of the same logits, and the logits match the oracle."""
    topk = cuda_lib
    n_q, n_kv, k = 16, 9000, 512
    starts = np.array([0, 100, 2000, 4000] * 4, np.int64)
    lens = np.array([9000, 5000, 7000, 600] * 4, np.int64)
    w = wl.indexer_inputs("cuda", 10, n_q=n_q, n_kv=n_kv, windows=(starts, starts + lens))
    stride = n_kv + 8
    logits = torch.full((n_q, stride), FILL, dtype=torch.float32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    seq_lens = (w["ke"] - w["ks"]).to(torch.int32)
    ws = topk.new_workspace(n_q, "cuda")
    out = torch.empty((n_q, k), dtype=torch.int32, device="cuda")
    out_raw = torch.empty((n_q, k), dtype=torch.int32, device="cuda")

    def step():
        topk.topk_indexer_logits(w["q"], w["kv"], w["kv_scale"], w["weights"], w["ks"], w["ke"], logits, stride, flags)
        topk.topk_plan(seq_lens, k, ws)
        topk.topk_transform_ragged(logits, stride, w["ks"], seq_lens, w["ks"], k, ws, out, out_raw,
                                   flags=topk.TOPK_DETERMINISTIC)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    # fresh inputs in the captured buffers, then replay
    fresh = wl.indexer_inputs("cuda", 11, n_q=n_q, n_kv=n_kv, windows=(starts, starts + lens))
    for key in ("q", "kv", "kv_scale", "weights"):
        w[key].copy_(fresh[key])
    logits.fill_(FILL)
    out.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    hw = host(w)
    got = logits.cpu().numpy()
    check_rows(got[[0, 5, 10, 15]], {**hw, "q": hw["q"][[0, 5, 10, 15]], "weights": hw["weights"][[0, 5, 10, 15]],
                                     "ks": hw["ks"][[0, 5, 10, 15]], "ke": hw["ke"][[0, 5, 10, 15]]},
               np.arange(4), 0, stride)
    tw = dict(mode="ragged", k=k, scores=logits.reshape(-1), score_stride=stride, row_starts=w["ks"],
              seq_lens=seq_lens, out_offsets=w["ks"], page_table=None, page_table_stride=0, page_size=1,
              batch=n_q, name="graph-replayed indexer logits -> ragged top-k")
    ref_out, ref_raw, err = oracle.run_workload(tw)
    assert err == 0
    compare_with_oracle(HostWorkload(tw), out.cpu().numpy(), out_raw.cpu().numpy(), ref_out, ref_raw,
                        deterministic=True)
