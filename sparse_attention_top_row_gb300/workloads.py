"""Seeded synthetic inputs for the indexer top-k + transform.

This module only draws random inputs; it holds none of the selection or
transform arithmetic. The tests feed the same tensors to the CUDA library and
to the CPU oracle, and the benchmark times the library on them.

Every generator takes a ``device`` (``"cpu"`` or ``"cuda"``) and a seed; a
seeded ``torch.Generator`` on that device draws the values, so a given
(device, seed) always yields the same bytes. Seeds follow
``20260000 + workload_id * 100 + sub_id``.

A workload is a plain dict:

    mode            "paged" | "ragged"
    k               int, 1..2048
    scores          float32 tensor; row b's window begins at element
                    b*score_stride + row_starts[b] of its flattened storage
    score_stride    int (elements; a multiple of 4, 0 = all rows share one buffer)
    row_starts      int32 [B] or None (None = every window starts at 0)
    seq_lens        int32 [B]
    out_offsets     int32 [B] (RAGGED) or None
    page_table      int32 [B, P] (PAGED) or None
    page_table_stride, page_size
    page_table_row_starts, row_to_batch
                    int32 [B] or absent (packed PAGED: the page-table lookup
                    of row b starts at request-local token
                    page_table_row_starts[b] of table row row_to_batch[b])
    batch           B
    name            short description

Scores outside every window hold the sentinel 1e3, so a window leak would win
the selection (the sentinel design of the sglang PR #35175 page's tests).
"""

from __future__ import annotations

import math

import torch

SENTINEL = 1.0e3
SEED_BASE = 20260000


def seed_for(workload_id: int, sub_id: int = 0) -> int:
    return SEED_BASE + workload_id * 100 + sub_id


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _i32(x):
    return x.to(torch.int32).contiguous()


def ragged_tiny(device="cpu", sub_id=0, batch=8, k=512, max_len=4096):
    """Eight windows packed back to back in one fp32 buffer (stride 0).

    seq_lens ~ U{1..max_len}; row_starts = exclusive prefix sum (so the
    residues mod 4 vary); out_offsets = row_starts; N(0,1) scores inside the
    windows; the 1e3 sentinel after the last window, padding the buffer to a
    multiple of 4 plus 64 floats of slack.
    """
    g = _gen(device, seed_for(1, sub_id))
    seq_lens = torch.randint(1, max_len + 1, (batch,), generator=g, device=device)
    starts = torch.zeros(batch, dtype=torch.int64, device=device)
    starts[1:] = torch.cumsum(seq_lens, 0)[:-1]
    total = int(seq_lens.sum().item())
    n = (total + 3) // 4 * 4 + 64
    scores = torch.full((n,), SENTINEL, dtype=torch.float32, device=device)
    scores[:total] = torch.randn(total, generator=g, device=device)
    return dict(name=f"ragged tiny B={batch} k={k}", mode="ragged", k=k, scores=scores,
                score_stride=0, row_starts=_i32(starts), seq_lens=_i32(seq_lens),
                out_offsets=_i32(starts), page_table=None, page_table_stride=0,
                page_size=1, batch=batch)


def paged_decode(device="cpu", sub_id=0, batch=128, seq_len=8192, k=2048, page_size=64):
    """[batch, seq_len] N(0,1) scores, one full window per row, and a page
    table holding a seeded random permutation of batch*seq_len/page_size
    physical pages."""
    g = _gen(device, seed_for(2, sub_id))
    scores = torch.randn(batch, seq_len, generator=g, device=device)
    pages = (seq_len + page_size - 1) // page_size
    table = torch.randperm(batch * pages, generator=g, device=device).view(batch, pages)
    seq_lens = torch.full((batch,), seq_len, dtype=torch.int32, device=device)
    return dict(name=f"paged decode B={batch} L={seq_len} k={k} ps={page_size}", mode="paged",
                k=k, scores=scores, score_stride=seq_len, row_starts=None, seq_lens=seq_lens,
                out_offsets=None, page_table=_i32(table), page_table_stride=pages,
                page_size=page_size, batch=batch)


def ragged_extend(device="cpu", chunk=0, rows_per_chunk=1024, n_req=4, prefix=28672, new=4096,
                  k=2048, outlier_frac=0.01, outlier_value=4.0, sub_id=None):
    """One chunk of a prefill-extend problem.

    ``n_req`` requests, each with a ``prefix``-token cached prefix and ``new``
    new tokens, give ``n_req*new`` causal query rows. Query i of request r has
    seq_len = prefix+i+1 and row_start = r*(prefix+new) in a flattened KV row
    space of n_req*(prefix+new) columns (the row stride). out_offsets =
    row_start. Window scores are N(0,1) with ``outlier_frac`` of them set to
    exactly ``outlier_value``; every other column holds the 1e3 sentinel.
    Chunk c covers global rows c*rows_per_chunk ... and is generated from its
    own seed (sub_id, default c), so any chunk can be drawn alone.
    """
    g = _gen(device, seed_for(3, chunk if sub_id is None else sub_id))
    stride = n_req * (prefix + new)
    rows = torch.arange(chunk * rows_per_chunk, (chunk + 1) * rows_per_chunk, device=device)
    req = rows // new
    qi = rows % new
    seq_lens = prefix + qi + 1
    starts = req * (prefix + new)
    cols = torch.arange(stride, device=device)
    inside = (cols[None, :] >= starts[:, None]) & (cols[None, :] < (starts + seq_lens)[:, None])
    vals = torch.randn(rows_per_chunk, stride, generator=g, device=device)
    outl = torch.rand(rows_per_chunk, stride, generator=g, device=device) < outlier_frac
    vals = torch.where(outl, torch.full_like(vals, outlier_value), vals)
    scores = torch.where(inside, vals, torch.full_like(vals, SENTINEL))
    del vals, outl, inside
    return dict(name=f"ragged extend chunk={chunk} rows={rows_per_chunk} req={n_req} "
                     f"prefix={prefix} new={new} k={k}",
                mode="ragged", k=k, scores=scores, score_stride=stride, row_starts=_i32(starts),
                seq_lens=_i32(seq_lens), out_offsets=_i32(starts), page_table=None,
                page_table_stride=0, page_size=1, batch=rows_per_chunk)


def ragged_swa(device="cpu", sub_id=0, n_req=2, prefix=28672, new=512, ratio=4, window=128, k=512):
    """Compressed-KV top-k rows with the sliding-window combine (the PR #30255
    page's SWA combine; the reading is the library's topk_transform_ragged_swa).

    Query i of request r sits at raw token position pos = prefix + i; its
    compressed window holds L = (pos + 1) // ratio entries starting at
    row_start = r * C in a compressed row space of C columns per request (the
    longest window rounded up past a multiple of 4); out_offsets = row_start, and the window tokens map
    through swa_offsets = r * (prefix + new) (the raw token space). Scores are
    N(0,1) inside the windows and the 1e3 sentinel elsewhere. The combined
    rows are k + window wide.
    """
    g = _gen(device, seed_for(8, sub_id))
    per_req = ((prefix + new) // ratio + 4) // 4 * 4  # > the longest window, a multiple of 4
    stride = n_req * per_req
    rows = torch.arange(n_req * new, device=device)
    req = rows // new
    pos = prefix + rows % new
    seq_lens = (pos + 1) // ratio
    starts = req * per_req
    cols = torch.arange(stride, device=device)
    inside = (cols[None, :] >= starts[:, None]) & (cols[None, :] < (starts + seq_lens)[:, None])
    vals = torch.randn(n_req * new, stride, generator=g, device=device)
    scores = torch.where(inside, vals, torch.full_like(vals, SENTINEL))
    del vals, inside
    return dict(name=f"ragged swa req={n_req} prefix={prefix} new={new} ratio={ratio} window={window} k={k}",
                mode="ragged", k=k, scores=scores, score_stride=stride, row_starts=_i32(starts),
                seq_lens=_i32(seq_lens), out_offsets=_i32(starts), page_table=None, page_table_stride=0,
                page_size=1, batch=n_req * new, positions=_i32(pos), window_size=window,
                swa_offsets=_i32(req * (prefix + new)), out_width=k + window)


def paged_long(device="cpu", sub_id=0, batch=1, seq_len=131072, k=2048, page_size=64, scale=0.1):
    """Few long PAGED rows whose scores are 0.1*N(0,1) rounded to
    bf16-representable values (heavy exact ties near the threshold)."""
    g = _gen(device, seed_for(4, sub_id))
    scores = (scale * torch.randn(batch, seq_len, generator=g, device=device))
    scores = scores.to(torch.bfloat16).to(torch.float32)
    pages = (seq_len + page_size - 1) // page_size
    table = torch.randperm(batch * pages, generator=g, device=device).view(batch, pages)
    seq_lens = torch.full((batch,), seq_len, dtype=torch.int32, device=device)
    return dict(name=f"paged long B={batch} L={seq_len} k={k} bf16 ties", mode="paged", k=k,
                scores=scores, score_stride=seq_len, row_starts=None, seq_lens=seq_lens,
                out_offsets=None, page_table=_i32(table), page_table_stride=pages,
                page_size=page_size, batch=batch)


def paged_packed(device="cpu", sub_id=0, n_req=4, q_rows=4, min_tokens=12000, max_tokens=40000, window=16384,
                 k=2048, page_size=64):
    """Packed PAGED rows (multi-query extend): ``n_req`` requests, the last
    ``q_rows`` tokens of each a query row.

    Request r holds T_r ~ U{min_tokens..max_tokens} tokens and its own page
    table row (a seeded random permutation over all requests' pages). Every
    query row's scores live in one flattened key space of all requests
    (stride = sum T_r): request r's keys at batch-global offset cu[r], N(0,1)
    there, the 1e3 sentinel elsewhere. Query token i of request r sees the
    sliding window of request-local tokens [max(0, i + 1 - window), i], so
    page_table_row_starts = that start, row_starts = cu[r] + the start,
    seq_len = its length, row_to_batch = r.
    """
    g = _gen(device, seed_for(6, sub_id))
    T = torch.randint(min_tokens, max_tokens + 1, (n_req,), generator=g, device=device)
    cu = torch.zeros(n_req + 1, dtype=torch.int64, device=device)
    cu[1:] = torch.cumsum(T, 0)
    stride = (int(cu[-1].item()) + 3) // 4 * 4
    B = n_req * q_rows
    rtb = torch.arange(n_req, device=device).repeat_interleave(q_rows)
    qi = torch.arange(q_rows, device=device).repeat(n_req)
    tok = T[rtb] - q_rows + qi                       # request-local token of each query
    pt_start = torch.clamp(tok + 1 - window, min=0)
    seq_lens = tok + 1 - pt_start
    row_starts = cu[:-1][rtb] + pt_start
    scores = torch.full((B, stride), SENTINEL, dtype=torch.float32, device=device)
    for b in range(B):
        r = int(rtb[b].item())
        a, e = int(cu[r].item()), int(cu[r + 1].item())
        scores[b, a:e] = torch.randn(e - a, generator=g, device=device)
    pages = (int(T.max().item()) + page_size - 1) // page_size
    table = torch.randperm(n_req * pages, generator=g, device=device).view(n_req, pages)
    return dict(name=f"paged packed {n_req} requests x {q_rows} queries k={k}", mode="paged", k=k,
                scores=scores, score_stride=stride, row_starts=_i32(row_starts), seq_lens=_i32(seq_lens),
                out_offsets=None, page_table=_i32(table), page_table_stride=pages, page_size=page_size,
                page_table_row_starts=_i32(pt_start), row_to_batch=_i32(rtb), batch=B)


BOUNDARY_LENGTHS = (8192, 8193, 16384, 16385, 65535, 65536, 65537)


def boundary_lengths(k):
    return (k, k + 1) + BOUNDARY_LENGTHS


def mixed(device="cpu", mode="paged", k=2048, batch=129, sub_id=0, max_len=131072, min_len=256,
          page_size=64, boundary=True, boundary_index=None):
    """Mixed-length sweep in one launch.

    seq_lens are log-uniform in [min_len, max_len]; rows 0..min(9,B)-1 are
    overwritten with the boundary lengths k, k+1, 8192, 8193, 16384, 16385,
    65535, 65536, 65537 (clipped to max_len). With ``boundary_index`` set the
    single row takes that boundary length. PAGED: stride max_len, windows start
    at 0, page table [B, max_len/page_size] = a random permutation. RAGGED:
    stride max_len+4, row_starts ~ U{0..3}, out_offsets = b*stride + row_start.
    N(0,1) inside windows, the 1e3 sentinel outside.
    """
    g = _gen(device, seed_for(5, sub_id))
    u = torch.rand(batch, generator=g, device=device, dtype=torch.float64)
    lo, hi = math.log(min_len), math.log(max_len)
    seq_lens = torch.round(torch.exp(lo + u * (hi - lo))).to(torch.int64)
    blen = [min(x, max_len) for x in boundary_lengths(k)]
    if boundary_index is not None:
        seq_lens[0] = blen[boundary_index]
    elif boundary:
        n = min(len(blen), batch)
        seq_lens[:n] = torch.tensor(blen[:n], device=device)
    if mode == "paged":
        stride = max_len
        starts = torch.zeros(batch, dtype=torch.int64, device=device)
    else:
        stride = max_len + 4
        starts = torch.randint(0, 4, (batch,), generator=g, device=device)
    cols = torch.arange(stride, device=device)
    inside = (cols[None, :] >= starts[:, None]) & (cols[None, :] < (starts + seq_lens)[:, None])
    vals = torch.randn(batch, stride, generator=g, device=device)
    scores = torch.where(inside, vals, torch.full_like(vals, SENTINEL))
    del vals, inside
    w = dict(name=f"mixed {mode} B={batch} k={k} max_len={max_len}", mode=mode, k=k,
             scores=scores, score_stride=stride, seq_lens=_i32(seq_lens), batch=batch,
             page_size=page_size)
    if mode == "paged":
        pages = (max_len + page_size - 1) // page_size
        table = torch.randperm(batch * pages, generator=g, device=device).view(batch, pages)
        w.update(row_starts=None, out_offsets=None, page_table=_i32(table),
                 page_table_stride=pages)
    else:
        offs = torch.arange(batch, device=device) * stride + starts
        w.update(row_starts=_i32(starts), out_offsets=_i32(offs), page_table=None,
                 page_table_stride=0, page_size=1)
    return w


def _e4m3_codes(x):
    """FP8 E4M3 codes (uint8) of a float tensor, rounded by torch's
    float8_e4m3fn conversion (input drawing only)."""
    return x.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()


def indexer_inputs(device="cpu", sub_id=0, n_q=13, n_kv=1000, windows=None, heads=64, dim=128):
    """Inputs of the indexer logits (the producer upstream of the top-k):
    q [n_q, heads, dim] and kv [n_kv, dim] as FP8 E4M3 codes of N(0, 2^2)
    draws, kv_scale [n_kv] ~ U(0.005, 0.02) (a dequantisation scale), weights
    [n_q, heads] ~ N(0, 1/64), and each query's key window [ks, ke): given,
    or drawn at random (empty, clamped and partial-tile windows included)."""
    g = _gen(device, seed_for(9, sub_id))
    q = _e4m3_codes(2.0 * torch.randn(n_q, heads, dim, generator=g, device=device))
    kv = _e4m3_codes(2.0 * torch.randn(n_kv, dim, generator=g, device=device))
    kv_scale = 0.005 + 0.015 * torch.rand(n_kv, generator=g, device=device)
    weights = torch.randn(n_q, heads, generator=g, device=device) / 8.0
    if windows is None:
        a = torch.randint(-40, n_kv + 40, (n_q,), generator=g, device=device)
        b = a + torch.randint(-5, n_kv + 80, (n_q,), generator=g, device=device)
        ks, ke = _i32(a), _i32(b)
    else:
        ks, ke = (torch.as_tensor(x, dtype=torch.int32, device=device) for x in windows)
    return dict(name=f"indexer logits n_q={n_q} n_kv={n_kv}", q=q, kv=kv, kv_scale=kv_scale,
                weights=weights.contiguous(), ks=ks, ke=ke, n_q=n_q, n_kv=n_kv)


def indexer_extend(device="cpu", chunk=0, rows_per_chunk=1024, n_req=4, prefix=28672, new=4096, sub_id=None):
    """The indexer logits feeding one chunk of the prefill-extend top-k:
    the same query rows and windows as ``ragged_extend`` (query i of request
    r: keys [r*(prefix+new), r*(prefix+new) + prefix + i + 1) of the
    flattened KV of n_req*(prefix+new) keys), with FP8 inputs drawn as in
    ``indexer_inputs``. The logits' row stride is the flattened KV length."""
    rows = torch.arange(chunk * rows_per_chunk, (chunk + 1) * rows_per_chunk, device=device)
    req = rows // new
    starts = req * (prefix + new)
    ends = starts + prefix + rows % new + 1
    w = indexer_inputs(device, chunk if sub_id is None else sub_id, n_q=rows_per_chunk,
                       n_kv=n_req * (prefix + new), windows=(starts, ends))
    w["name"] = f"indexer logits, extend chunk={chunk} rows={rows_per_chunk} req={n_req} prefix={prefix} new={new}"
    w["stride"] = n_req * (prefix + new)
    return w


def custom(mode, k, rows, *, device="cpu", score_stride=None, row_starts=None, out_offsets=None,
           page_size=1, page_table=None, seed=0):
    """Build a workload from explicit per-row score lists (small edge cases).

    ``rows`` is a list of float lists; row b's window is rows[b] placed at
    row_starts[b] (default 0) of a row of ``score_stride`` elements (default:
    the longest window + start, rounded up to a multiple of 4). Outside the
    windows the sentinel is stored. PAGED without a table gets a seeded random
    permutation.
    """
    B = len(rows)
    starts = list(row_starts) if row_starts is not None else [0] * B
    need = max([s + len(r) for s, r in zip(starts, rows)] + [1])
    if score_stride is None:
        score_stride = (need + 3) // 4 * 4
    flat = torch.full((max(B, 1) * score_stride + 64,), SENTINEL, dtype=torch.float32)
    for b, (s, r) in enumerate(zip(starts, rows)):
        if len(r):
            base = b * score_stride + max(s, 0)
            flat[base:base + len(r)] = torch.tensor(r, dtype=torch.float32)
    seq_lens = torch.tensor([len(r) for r in rows], dtype=torch.int32)
    w = dict(name="custom", mode=mode, k=k, scores=flat.to(device), score_stride=score_stride,
             seq_lens=seq_lens.to(device), batch=B, page_size=page_size,
             row_starts=torch.tensor(starts, dtype=torch.int32, device=device)
             if row_starts is not None else None)
    if mode == "paged":
        pages = max((need + page_size - 1) // page_size, 1)
        if page_table is None:
            g = _gen("cpu", seed)
            page_table = torch.randperm(B * pages, generator=g).view(B, pages)
        page_table = torch.as_tensor(page_table, dtype=torch.int32)
        w.update(page_table=page_table.contiguous().to(device),
                 page_table_stride=int(page_table.shape[1]), out_offsets=None)
    else:
        offs = out_offsets if out_offsets is not None else [0] * B
        w.update(out_offsets=torch.tensor(offs, dtype=torch.int32, device=device),
                 page_table=None, page_table_stride=0)
    return w


def pack_windows(w):
    """The same rows with only their windows kept, packed back to back in one
    flat buffer: score_stride 0, row_starts = the exclusive prefix sum of
    seq_lens (so the starts' residues mod 4 vary), every other array as in
    ``w``. This is the input a caller that holds just the windows would move;
    RAGGED outputs (position + out_offsets[b]) and PAGED outputs (positions
    count from the window start) are the same as for ``w``. The 1e3 sentinel
    pads the tail to a multiple of 4 floats plus 64. Needs seq_lens >= 0 and
    row_starts >= 0; works on any device."""
    dev = w["seq_lens"].device
    B = int(w["batch"])
    lens = w["seq_lens"].to(torch.int64)
    if bool((lens < 0).any()):
        raise ValueError("pack_windows needs non-negative seq_lens")
    starts = (w["row_starts"].to(torch.int64) if w.get("row_starts") is not None
              else torch.zeros(B, dtype=torch.int64, device=dev))
    flat = w["scores"].reshape(-1)
    total = int(lens.sum().item())
    new_starts = torch.cumsum(lens, 0) - lens
    row_of = torch.repeat_interleave(torch.arange(B, device=dev), lens)
    src = (row_of * int(w["score_stride"]) + starts[row_of] +
           torch.arange(total, device=dev) - new_starts[row_of])
    packed = torch.full(((total + 3) // 4 * 4 + 64,), SENTINEL, dtype=torch.float32, device=dev)
    packed[:total] = flat[src]
    del src, row_of
    out = dict(w)
    out.update(scores=packed, score_stride=0, row_starts=_i32(new_starts),
               name=w["name"] + " (windows packed)")
    return out


def to_device(w, device):
    """Copy every tensor of a workload to ``device``."""
    return {key: (val.to(device) if isinstance(val, torch.Tensor) else val) for key, val in w.items()}


def select_rows(w, rows):
    """A workload holding only ``rows`` of ``w`` (each row's slice of the
    score storage is copied, with the sentinel-filled remainder of its
    stride). Stride-0 workloads keep the whole shared buffer."""
    rows = [int(r) for r in rows]
    idx = torch.tensor(rows, dtype=torch.long, device=w["seq_lens"].device)
    stride = int(w["score_stride"])
    flat = w["scores"].reshape(-1)
    if stride == 0:
        scores = flat.clone()
    else:
        scores = torch.stack([flat[r * stride:(r + 1) * stride] for r in rows]).reshape(-1)
    out = dict(w)
    out.update(scores=scores, batch=len(rows), seq_lens=w["seq_lens"][idx].clone(),
               name=w["name"] + f" rows={rows[:4]}...")
    for key in ("row_starts", "out_offsets", "page_table_row_starts", "row_to_batch", "positions", "swa_offsets"):
        if w.get(key) is not None:
            out[key] = w[key][idx].clone()
    if w.get("page_table") is not None and w.get("row_to_batch") is None:
        out["page_table"] = w["page_table"][idx].clone()  # packed rows keep the request tables
    return out


def shard_rows(w, rank, world):
    """Rank `rank`'s contiguous block of the batch's rows when the rows are
    partitioned over `world` GPUs (rows are independent: each GPU needs only
    its rows' scores, lengths, starts, offsets and page-table rows, and no
    exchange follows). Block r holds rows [r*B//world, (r+1)*B//world)."""
    B = int(w["batch"])
    lo, hi = rank * B // world, (rank + 1) * B // world
    return select_rows(w, range(lo, hi)) if hi > lo else None
