#!/usr/bin/env python3
"""Benchmark of the indexer top-k + transform on GB300.

One step = the whole hot path on one batch: topk_plan + the transform
(route, 16-byte window loads, key map, histogram threshold search, radix
refine, compaction, fused page-table / offset emit).

Headline workload: RAGGED prefill extend, 4 requests x (28672 cached + 4096
new tokens) = 16384 causal query rows of 28673..32768 fp32 scores, k = 2048,
out_offsets = row_start, stored as a [16384, 131072] fp32 buffer and run as 16
launches of 1024 rows. Its 8 GiB of scores span far more than twice the L2, so
no timed step finds its inputs there. The other workloads (RAGGED tiny, PAGED
decode, PAGED long, packed PAGED, the mixed sweep) are measured after it and
reported under "configs"; those small enough to fit in L2 are rotated through
at least ceil(2 * L2 / set bytes) + 1 copies of their inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU with
its own seed (weak scaling; rows are independent, so there is no data-path
collective); the barrier and the max-over-ranks time use torch.distributed.
``--impl reference`` times the CPU oracle, as it stands, on the host cores
(every core, each thread running the unchanged single-threaded routine on its
own block of rows): W untimed steps, then K timed steps, each a bounded
sample of the headline workload's rows.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import sparse_attention_top_row_gb300 as topk  # noqa: E402
from sparse_attention_top_row_gb300 import workloads as wl  # noqa: E402

METRIC = "rows/sec and achieved HBM GB/s (fraction of ~8 TB/s) for top-k transform, 1×GB300"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 126 * 1024 * 1024
HEADLINE = "ragged_extend"
REF_BUDGET_S = 120.0     # the whole reference-arm run, warm-up included
MAX_ROTATION_BYTES = 6 << 30   # device memory a rotation of small input sets may take
KERNEL_SRCS = [os.path.join(ROOT, "sparse_attention_top_row_gb300", "csrc", f)
               for f in ("topk.cu", "topk_common.cuh", "topk_select.cuh", "topk_select512.cu", "topk_select256.cu")]


# ----------------------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


LOGITS_SRCS = [os.path.join(ROOT, "sparse_attention_top_row_gb300", "csrc", f)
               for f in ("topk_logits.cu", "topk_common.cuh")]


def kernel_source_hash(srcs=None):
    """First 16 hex digits of the SHA-256 of the kernel sources, concatenated
    (the selection kernels' by default)."""
    h = hashlib.sha256()
    for path in srcs or KERNEL_SRCS:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload, srcs=None):
    """DRAM bytes (read + written) per launch of `kernel` on `workload` from
    the committed ncu record ``profiles/<kernel>_<workload>.json``, if that
    record was taken on the current kernel source (`srcs`, the selection
    kernels' by default); else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel_source_sha256_16") != kernel_source_hash(srcs):
        return None
    return int(rec["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- workloads

DESCRIPTIONS = {
    "ragged_extend": "RAGGED prefill extend: 4 requests x (28672 cached + 4096 new) = 16384 causal rows, "
                     "L = 28673..32768, k=2048, out_offsets = row_start, [16384, 131072] fp32 run as 16 "
                     "launches of 1024 rows; N(0,1) with 1% +4.0",
    "ragged_tiny": "RAGGED tiny: B=8, k=512, L ~ U{1..4096}, windows back to back in one buffer",
    "paged_decode": "PAGED decode: B=128, L=8192, k=2048, page_size=64, random page permutation",
    "paged_long_b1": "PAGED long: B=1, L=131072, k=2048, page_size=64, bf16-rounded 0.1*N(0,1)",
    "paged_long_b30": "PAGED long: B=30, L=131072, k=2048, page_size=64, bf16-rounded 0.1*N(0,1)",
    "paged_long_b31": "PAGED long: B=31, L=131072, k=2048, page_size=64, bf16-rounded 0.1*N(0,1)",
    "paged_packed": "packed PAGED: 8 requests x 16 query rows, sliding window 16384, k=2048, page_size=64",
    "mixed": "mixed sweep: k in {512,1024,2048} x B in {1,31,129,1024} x {PAGED, RAGGED}, "
             "L log-uniform in [256, 131072] plus boundary rows (24 launches)",
    "ragged_swa": "RAGGED top-k fused with the SWA combine: 4 requests x 1024 queries at positions 28672.., "
                  "compressed windows of (pos+1)//4 = 7168..7424 entries, k=512, window 128, rows of 640",
}
EXTRA = ("ragged_tiny", "paged_decode", "paged_long_b1", "paged_long_b30", "paged_long_b31", "paged_packed",
         "mixed", "ragged_swa")


def make_workload(name, device, rank=0):
    """The named workload as a list of launches (each a workload dict)."""
    if name == "paged_decode":
        return [wl.paged_decode(device, sub_id=rank)]
    if name == "ragged_tiny":
        return [wl.ragged_tiny(device, sub_id=rank)]
    if name == "ragged_extend":
        return [wl.ragged_extend(device, chunk=c, sub_id=c + 16 * rank) for c in range(16)]
    if name == "ragged_swa":  # compressed-KV top-k fused with the sliding-window combine
        return [wl.ragged_swa(device, sub_id=rank, n_req=4, new=1024, prefix=28672, ratio=4, window=128, k=512)]
    if name == "ragged_extend_chunk":  # one 1024-row chunk (profiling size)
        return [wl.ragged_extend(device, chunk=0)]
    if name == "paged_packed":  # packed PAGED extend rows: 8 requests x 16 queries, sliding window 16384
        return [wl.paged_packed(device, sub_id=rank, n_req=8, q_rows=16)]
    if name.startswith("paged_long_b"):
        b = int(name[len("paged_long_b"):])
        return [wl.paged_long(device, batch=b, sub_id=b + 100 * rank)]
    if name == "mixed":
        launches = []
        for mode in ("paged", "ragged"):
            for k in (512, 1024, 2048):
                for b in (1, 31, 129, 1024):
                    launches.append(wl.mixed(device, mode=mode, k=k, batch=b, sub_id=b + 100 * rank))
        return launches
    raise ValueError(name)


def headline_sample(device="cpu"):
    """The bounded sample of the headline workload the CPU oracle is timed on:
    rows 2048..2303 of the 16384 (query tokens 2048..2303 of request 0, L =
    30721..30976, about the workload's mean length of 30720.5), drawn by the
    same recipe from their own seed."""
    return wl.ragged_extend(device, chunk=8, rows_per_chunk=256)


def algorithmic_bytes(w, out_raw):
    """Scores read by non-trivial rows + indices written + distinct page-table
    entries read + 4 B per per-row array read."""
    k = int(w["k"])
    lens = w["seq_lens"].to(torch.int64).clamp(min=0)
    nontrivial = lens > k
    scores = int((4 * lens[nontrivial]).sum().item())
    swa = w.get("positions") is not None  # the fused SWA combine writes rows of out_width
    out = 4 * (int(w["out_width"]) if swa else k) * int(w["batch"])
    packed = [w.get(key) for key in ("page_table_row_starts", "row_to_batch")]
    if swa:
        packed += [w["positions"], w.get("swa_offsets")]
    meta = 4 * int(w["batch"]) * (1 + (w.get("row_starts") is not None) + (w["mode"] == "ragged") +
                                  sum(a is not None for a in packed))
    pages = 0
    if w["mode"] == "paged":
        ps = int(w["page_size"])
        r = out_raw.to(torch.int64)
        if packed[0] is not None:  # packed rows read their tables from token page_table_row_starts[b]
            r = torch.where(r >= 0, r + packed[0].to(torch.int64)[:, None], r)
        pg = torch.where(r >= 0, r // ps, torch.full_like(r, -1))
        srt, _ = torch.sort(pg, dim=1)
        distinct = ((srt[:, 1:] != srt[:, :-1]) & (srt[:, 1:] >= 0)).sum(1) + (srt[:, 0] >= 0).to(torch.int64)
        pages = 4 * int(distinct.sum().item())
    return scores + out + meta + pages


def input_bytes(w):
    return sum(v.numel() * v.element_size() for v in w.values() if isinstance(v, torch.Tensor))


def transform_kernels(batch):
    """Kernels one transform of `batch` rows launches (the library's own
    count for the current device)."""
    return topk.topk_transform_launches(batch)


class Launch:
    """Device buffers + workspace for one launch, and its step function."""

    def __init__(self, w, flags=0):
        self.w = w
        self.B, self.k = int(w["batch"]), int(w["k"])
        self.swa = w.get("positions") is not None  # the fused SWA combine: rows of out_width
        width = int(w["out_width"]) if self.swa else self.k
        self.out = torch.empty((self.B, width), dtype=torch.int32, device=w["scores"].device)
        self.ws = topk.new_workspace(self.B, w["scores"].device)
        self.flags = flags

    def plan(self, stream):
        topk.topk_plan(self.w["seq_lens"], self.k, self.ws, stream=stream)

    def transform(self, stream, out_raw=None):
        w = self.w
        if w["mode"] == "paged" and w.get("row_to_batch") is not None:
            topk.topk_transform_paged_packed(w["scores"], w["score_stride"], w.get("row_starts"), w["seq_lens"],
                                             w["page_table"], w["page_table_stride"], w["page_size"],
                                             w.get("page_table_row_starts"), w["row_to_batch"], self.k,
                                             self.ws, self.out, out_raw, self.flags, stream=stream)
        elif w["mode"] == "paged":
            topk.topk_transform_paged(w["scores"], w["score_stride"], w.get("row_starts"), w["seq_lens"],
                                      w["page_table"], w["page_table_stride"], w["page_size"], self.k,
                                      self.ws, self.out, out_raw, self.flags, stream=stream)
        elif self.swa:
            topk.topk_transform_ragged_swa(w["scores"], w["score_stride"], w.get("row_starts"), w["seq_lens"],
                                           w["out_offsets"], self.k, self.ws, w["positions"], w["window_size"],
                                           w.get("swa_offsets"), w["out_width"], self.out, out_raw, self.flags,
                                           stream=stream)
        else:
            topk.topk_transform_ragged(w["scores"], w["score_stride"], w.get("row_starts"), w["seq_lens"],
                                       w["out_offsets"], self.k, self.ws, self.out, out_raw, self.flags,
                                       stream=stream)

    def launches_per_step(self):
        return 1 + transform_kernels(self.B)


# ----------------------------------------------------------------------------- device timing

class L2Flush:
    """A device buffer of twice the L2; writing it evicts whatever the L2
    held (done outside every timed region)."""

    def __init__(self, l2_bytes):
        self.buf = torch.empty(2 * l2_bytes // 4 + 1024, dtype=torch.int32, device="cuda")

    def __call__(self, stream):
        with torch.cuda.stream(stream):
            self.buf.fill_(1)


def time_workload(launch_sets, steps, warmup, world, stream, flush):
    """Times `steps` steps; timed step i runs every launch of set
    (warmup + i) % len(sets). The steps are captured into one CUDA graph (the
    way a serving loop launches them), so the device timeline holds no host
    launch gaps; a second graph of the transforms alone gives the per-launch
    duration of the transform. The L2 is flushed before each of the two
    replays, and the sets a replay cycles through span more than twice the
    L2. Returns (seconds for all steps, seconds per transform launch)."""
    n_launch = len(launch_sets[0])

    def sets_for(i):
        return launch_sets[(warmup + i) % len(launch_sets)]

    for i in range(warmup):
        for ln in launch_sets[i % len(launch_sets)]:
            ln.plan(stream)
            ln.transform(stream)
    for i in range(steps):  # every workspace planned once before capture
        for ln in sets_for(i):
            ln.plan(stream)
    torch.cuda.synchronize()
    g_steps = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_steps):
        for i in range(steps):
            for ln in sets_for(i):
                ln.plan(None)
                ln.transform(None)
    g_tr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_tr):
        for i in range(steps):
            for ln in sets_for(i):
                ln.transform(None)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    flush(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev[0].record(stream)
    g_steps.replay()
    ev[1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    flush(stream)                   # the transforms alone, on cold inputs too
    ev[2].record(stream)
    g_tr.replay()
    ev[3].record(stream)
    torch.cuda.synchronize()
    total = ev[0].elapsed_time(ev[1]) / 1e3
    per_transform = ev[2].elapsed_time(ev[3]) / 1e3 / (steps * n_launch)
    del g_steps, g_tr
    return total, per_transform


def rotating_sets(name, device, rank, l2_bytes, flags=0):
    """Copies of a workload's inputs such that the sets span more than twice
    the L2: one set when it alone does, else ceil(2 * L2 / set bytes) + 1
    sets (capped by MAX_ROTATION_BYTES), whatever the step count."""
    base = make_workload(name, device, rank)
    size = sum(input_bytes(w) for w in base)
    n = 1 if size > 2 * l2_bytes else int(math.ceil(2 * l2_bytes / max(size, 1))) + 1
    n = max(1, min(n, MAX_ROTATION_BYTES // max(size, 1)))
    sets = [[Launch(w, flags) for w in base]]
    for c in range(1, n):
        sets.append([Launch({kk: (v.clone() if isinstance(v, torch.Tensor) else v) for kk, v in w.items()},
                            flags) for w in base])
    return sets, n, size


def measure(name, steps, warmup, world, rank, stream, peak, l2_bytes, flush):
    sets, n_sets, set_bytes = rotating_sets(name, "cuda", rank, l2_bytes)
    # algorithmic bytes, from one run with out_raw
    alg = 0
    for ln in sets[0]:
        raw = torch.empty_like(ln.out)
        ln.plan(stream)
        ln.transform(stream, out_raw=raw)
        torch.cuda.synchronize()
        alg += algorithmic_bytes(ln.w, raw)
    rows = sum(ln.B for ln in sets[0])
    total, t_launch = time_workload(sets, steps, warmup, world, stream, flush)
    total = max_over_ranks(total, world)
    t_transform = t_launch * len(sets[0])
    res = {
        "rows_per_s": world * rows * steps / total,
        "us_per_step": 1e6 * total / steps,
        "us_transform_per_step": 1e6 * t_transform,
        "alg_bytes_per_step": alg,
        "gbs_transform": alg / t_transform / 1e9,
        "frac_of_measured_hbm": alg / t_transform / 1e9 / peak,
        "frac_of_nominal_8tbs": alg / t_transform / 1e9 / NOMINAL_HBM_GBS,
        "input_sets": n_sets,
        "input_set_bytes": set_bytes,
        "l2": l2_text(n_sets, set_bytes, l2_bytes),
        "launches_per_step": sum(ln.launches_per_step() for ln in sets[0]),
        "rows_per_step": rows,
        "steps": steps,
    }
    del sets
    torch.cuda.empty_cache()
    return res


def l2_text(n_sets, set_bytes, l2_bytes):
    ok = n_sets * set_bytes >= 2 * l2_bytes
    return (f"{n_sets} input set(s) x {set_bytes} B = {n_sets * set_bytes} B "
            f"{'>=' if ok else '<'} 2 x L2 = {2 * l2_bytes} B; L2 flushed before each timed replay")


# ----------------------------------------------------------------------------- end to end

def packed_inputs(w, device):
    """The workload's input tensors packed into one pinned host buffer and one
    device buffer of the same layout (each tensor at a 256-byte offset), so a
    step moves all inputs with one host-to-device copy. Returns the pinned
    buffer, the device buffer and the workload with device views."""
    items = [(kk, v) for kk, v in w.items() if isinstance(v, torch.Tensor)]
    offs, total = [], 0
    for _, v in items:
        offs.append(total)
        total += -(-(v.numel() * v.element_size()) // 256) * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev = torch.empty(total, dtype=torch.uint8, device=device)
    out = dict(w)
    for (kk, v), off in zip(items, offs):
        n = v.numel() * v.element_size()
        host[off:off + n].copy_(v.contiguous().reshape(-1).view(torch.uint8))
        out[kk] = dev[off:off + n].view(v.dtype).view(v.shape)
    return host, dev, out


def e2e_host_workloads(name, rank):
    """Host copies of the workload's launches for the end-to-end leg. Rows
    whose score windows sit in a wider strided buffer keep only their windows,
    packed back to back (the bytes a caller actually holds and moves; outputs
    are unchanged: RAGGED positions get out_offsets[b], PAGED positions count
    from the window start)."""
    hosts = []
    devs = make_workload(name, "cuda", rank)
    for w in devs:
        windows = int(w["seq_lens"].clamp(min=0).sum().item())
        if int(w["score_stride"]) > 0 and w["scores"].numel() > 2 * windows:
            w = wl.pack_windows(w)
        hosts.append(wl.to_device(w, "cpu"))
    del devs
    torch.cuda.empty_cache()
    return hosts


def measure_e2e(name, steps, warmup, rank, stream):
    """Same metric through the public API with HOST buffers: each step copies
    every launch's inputs from pinned host memory (one packed copy per
    launch), plans, transforms and reads the output back to pinned host
    memory; the timed region holds all of it. The input copies run on a copy
    stream one launch ahead of the compute stream (launch i computes once its
    copy is in; its buffer is refilled only after the previous step's launch i
    is done), so the copies, which bound the step, overlap the kernels."""
    hosts = e2e_host_workloads(name, rank)
    packs = [packed_inputs(w, "cuda") for w in hosts]
    h2d = sum(hb.numel() for hb, _, _ in packs)
    d2h = sum(4 * int(w["batch"]) * int(w["k"]) for w in hosts)
    launches = [Launch(dw) for _, _, dw in packs]
    outs = [torch.empty((ln.B, ln.k), dtype=torch.int32).pin_memory() for ln in launches]
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in packs]
    done = [torch.cuda.Event() for _ in packs]
    for ev in done:
        ev.record(stream)

    def step():
        for i, ((hb, db, _), ln, ho) in enumerate(zip(packs, launches, outs)):
            copy_stream.wait_event(done[i])  # launch i of the previous step has read its buffer
            with torch.cuda.stream(copy_stream):
                db.copy_(hb, non_blocking=True)
            copied[i].record(copy_stream)
            stream.wait_event(copied[i])
            ln.plan(stream)
            ln.transform(stream)
            ho.copy_(ln.out, non_blocking=True)
            done[i].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        copy_stream.wait_event(a)
        for _ in range(steps):
            step()
        b.record(stream)  # after the last launch, which waited for the last copy
        torch.cuda.synchronize()
    t = a.elapsed_time(b) / 1e3
    # One more step, untimed and in deterministic mode (a unique result), read
    # back to the host: sampled rows of every launch must match the oracle.
    for ln in launches:
        ln.flags = topk.TOPK_DETERMINISTIC
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    import oracle
    for w, ho in zip(hosts, outs):
        B = int(w["batch"])
        rows = sorted({0, B // 3, B // 2, B - 1})
        ref, _, _ = oracle.run_workload(w, rows=rows)
        got = torch.sort(ho[rows], dim=1).values.numpy()
        if not (got == __import__("numpy").sort(ref, axis=1)).all():
            raise RuntimeError(f"end-to-end outputs differ from the oracle on {w['name']}")
    rows = sum(ln.B for ln in launches)
    res = {"value": rows * steps / t, "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": 1e3 * t / steps}
    del packs, launches, outs
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample(name, rank):
    """Host copies of a bounded row sample of every launch of the workload
    (up to 64 evenly spaced rows each; the headline's sample is
    headline_sample())."""
    if name == HEADLINE:
        return [headline_sample("cpu")], "rows 2048..2303 of the 16384 (L 30721..30976), their own seed"
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    out = []
    for w in make_workload(name, dev, rank):
        B = int(w["batch"])
        rows = sorted({int(round(i * (B - 1) / 63)) for i in range(64)}) if B > 64 else list(range(B))
        out.append(wl.to_device(wl.select_rows(w, rows) if len(rows) < B else w, "cpu"))
    return out, "up to 64 evenly spaced rows of every launch"


def time_oracle(samples, threads, budget_s):
    """Rows per second of the oracle, as it stands, over repeated passes of
    the sample (whole passes, at least one) until `budget_s` has passed; with
    threads > 1 every launch's rows are split over that many threads, each
    running the unchanged single-threaded routine. Returns (rows/s, rows,
    seconds)."""
    import oracle
    rows, t0 = 0, time.perf_counter()
    while True:
        for w in samples:
            oracle.run_workload_threads(w, threads=threads)
            rows += int(w["batch"])
        t = time.perf_counter() - t0
        if t >= budget_s:
            return rows / t, rows, t


def cpu_baselines(name, rank, budget_s):
    """The CPU oracle on one thread and on every host core."""
    import oracle
    samples, what = oracle_sample(name, rank)
    cores = oracle.host_cores()
    v1, r1, t1 = time_oracle(samples, 1, budget_s)
    vn, rn, tn = time_oracle(samples, cores, budget_s)
    return {"value": vn, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{what} of the {name} workload: {rn} rows in {tn:.1f} s on {cores} threads",
            "single_thread": {"value": v1, "unit": "rows/s", "cores": 1,
                              "sample": f"{r1} rows in {t1:.1f} s on 1 thread"}}


# ----------------------------------------------------------------------------- indexer logits

FP8_PER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor rates (4.5 / 2.25 PFLOP/s)


def measured_bf16_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def logits_flops(w):
    """Algorithmic FLOPs of the indexer logits: 2 * 64 * 128 per (query,
    key) pair inside a window (the head weighting and ReLU not counted)."""
    lens = (w["ke"].clamp(max=w["n_kv"]) - w["ks"].clamp(min=0)).clamp(min=0)
    return float(lens.to(torch.float64).sum()) * 2 * topk.TOPK_INDEXER_HEADS * topk.TOPK_INDEXER_DIM


def logits_cpu_baseline(budget_s):
    """The oracle's indexer logits, as it stands, on a bounded sample of the
    extend chunk: query rows 0, 1, ... over the first 256 keys of their
    windows, repeated until the budget has passed (one thread)."""
    import numpy as np

    import oracle
    w = wl.indexer_extend("cpu", 0)
    q, kv = w["q"].numpy(), w["kv"].numpy()
    scale, wt = w["kv_scale"].numpy(), w["weights"].numpy()
    ks = w["ks"].numpy()
    pairs, t0, i = 0, time.perf_counter(), 0
    out = np.zeros((1, w["stride"]), np.float32)
    while True:
        t = i % w["n_q"]
        lo = int(ks[t])
        oracle.indexer_logits(q[t:t + 1], kv, scale, wt[t:t + 1], [lo], [lo + 256], out)
        pairs += 256
        i += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            flops = pairs * 2.0 * topk.TOPK_INDEXER_HEADS * topk.TOPK_INDEXER_DIM
            return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                    "sample": f"{i} query rows x 256 keys of the extend chunk's windows in {el:.1f} s on 1 thread "
                              f"({pairs / el:.0f} logits/s)"}


def measure_logits(steps, warmup, stream, flush):
    """The indexer logits of one extend chunk (1024 queries over their
    windows of 28673..29696 keys in the 131072-key flattened KV), alone and
    fed straight into the RAGGED top-k of the same rows (plan + transform
    after it on the stream; the chunk's logits, 122 MB written, are read back
    mostly from L2). Both timed as CUDA graphs of `steps` repetitions, the L2
    flushed before each replay."""
    w = wl.indexer_extend("cuda", 0)
    stride, n_q = w["stride"], w["n_q"]
    logits = torch.full((n_q, stride), wl.SENTINEL, dtype=torch.float32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    flops = logits_flops(w)

    def produce():
        topk.topk_indexer_logits(w["q"], w["kv"], w["kv_scale"], w["weights"], w["ks"], w["ke"], logits, stride,
                                 flags)

    tw = dict(mode="ragged", k=2048, scores=logits, score_stride=stride, row_starts=w["ks"],
              seq_lens=(w["ke"] - w["ks"]).to(torch.int32), out_offsets=w["ks"], page_table=None,
              page_table_stride=0, page_size=1, batch=n_q, name="indexer logits -> top-k")
    ln = Launch(tw)
    for _ in range(warmup):
        produce()
        ln.plan(stream)
        ln.transform(stream)
    torch.cuda.synchronize()
    graphs = []
    for chain in (False, True):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(steps):
                produce()
                if chain:
                    ln.plan(None)
                    ln.transform(None)
        graphs.append(g)
    torch.cuda.synchronize()
    times = []
    for g in graphs:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        flush(stream)
        torch.cuda.synchronize()
        ev[0].record(stream)
        g.replay()
        ev[1].record(stream)
        torch.cuda.synchronize()
        times.append(ev[0].elapsed_time(ev[1]) / 1e3 / steps)
    assert int(flags.item()) == 0, "a bounded wait in the logits kernel gave up"
    t_logits, t_chain = times
    bf16, kind = measured_bf16_tflops()
    peak = bf16 * FP8_PER_BF16
    achieved = flops / t_logits / 1e12
    del graphs
    return {
        "workload": "indexer logits (FP8 E4M3 q [1024, 64, 128], kv [131072, 128], fp32 head weights) of one "
                    "RAGGED extend chunk: query i of request r over keys [32768 r, 32768 r + 28673 + i); then the "
                    "RAGGED top-k (k = 2048) of the same rows",
        "tflops": achieved,
        "us_per_launch": 1e6 * t_logits,
        "flops_per_launch": flops,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "dtype": "fp8 e4m3 (fp32 accumulate)",
                     "traffic": profiled_traffic("topk_indexer_logits_kernel", "indexer_logits_extend_chunk",
                                                 LOGITS_SRCS),
                     "peak_kind": f"{kind} bf16 burst x {FP8_PER_BF16} (nominal fp8/bf16 ratio)",
                     "kernel": "topk_indexer_logits_kernel (tcgen05.mma kind::f8f6f4, TMEM accumulators, TMA)"},
        "chain_us_per_step": 1e6 * t_chain,
        "chain_rows_per_s": n_q / t_chain,
        "chain": "logits -> plan -> RAGGED transform per step (3 launches, programmatic dependent launch)",
        "launches_per_step": 1,
        "l2": "inputs 25 MB (the 16.8 MB KV is meant to stay in L2: every query of a request reads it); "
              "output 512 MB buffer > 2 x L2; L2 flushed before each timed replay",
    }


# ----------------------------------------------------------------------------- main

def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on every host core
    (each thread running the unchanged single-threaded routine on its own
    block of rows) over a bounded sample of the headline workload. W untimed
    steps, then exactly K timed steps; a step is the oracle over R rows of
    the sample, R chosen from the first warm-up step so that the whole run
    stays within about REF_BUDGET_S. Rank 0 alone runs it."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    w = headline_sample("cpu")
    cores = oracle.host_cores()
    B = int(w["batch"])
    t0 = time.perf_counter()
    oracle.run_workload_threads(w, threads=cores)          # the first warm-up step, every sample row
    t_row = (time.perf_counter() - t0) / B
    n_steps = args.steps + args.warmup
    rows_per_step = max(1, min(B, int(REF_BUDGET_S / max(t_row * n_steps, 1e-9))))
    rows = np.arange(rows_per_step)
    for _ in range(args.warmup - 1):
        oracle.run_workload_threads(w, rows=rows, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run_workload_threads(w, rows=rows, threads=cores)
    t = time.perf_counter() - t0
    value = rows_per_step * args.steps / t
    base = {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{args.steps} timed step(s) after {args.warmup} warm-up step(s), each the oracle over "
                      f"{rows_per_step} of rows 2048..2303 (L 30721..30976) of the {HEADLINE} workload "
                      f"on {cores} threads"}
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)", "impl": "reference",
        "config": headline_config(world or 1),
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def headline_config(world, l2=None):
    cfg = {"workload": DESCRIPTIONS[HEADLINE], "global_batch": 16384 * world, "seq_len": "28673..32768",
           "k": 2048, "parallelism": f"rows x{world} (weak)"}
    if l2 is not None:
        cfg["l2"] = l2
    return cfg


def device_l2_bytes():
    try:
        return max(int(torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size),
                   126 * 1024 * 1024)
    except (RuntimeError, AttributeError):
        return 126 * 1024 * 1024


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-configs", action="store_true", help="headline workload only")
    ap.add_argument("--workload", default=HEADLINE,
                    help="the workload of a --quick run (a top-k workload, or indexer_logits)")
    ap.add_argument("--quick", action="store_true",
                    help="one workload only: device timings, no e2e, no CPU baseline")
    ap.add_argument("--cpu-seconds", type=float, default=1.5, help="oracle time budget per config and thread count")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        if world > 1:
            dist.destroy_process_group()
        return

    topk.load()
    peak, peak_kind = measured_peaks()
    stream = torch.cuda.current_stream()
    l2 = device_l2_bytes()
    flush = L2Flush(l2)

    name = args.workload if args.quick else HEADLINE
    if args.quick and name == "indexer_logits":
        with ClockSampler(local) as clocks:
            res = measure_logits(args.steps, args.warmup, stream, flush)
        if rank == 0:
            print(json.dumps({"workload": name, **res, "clocks": clocks.summary()}), flush=True)
        return
    with ClockSampler(local) as clocks:
        head = measure(name, args.steps, args.warmup, world, rank, stream, peak, l2, flush)
    clk = clocks.summary()
    if args.quick:
        if rank == 0:
            print(json.dumps({"workload": name, **head, "clocks": clk}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    e2e = measure_e2e(HEADLINE, args.steps, args.warmup, rank, stream)
    base = cpu_baselines(HEADLINE, rank, 3 * args.cpu_seconds) if (rank == 0 and world == 1) else None

    extra = {}
    if not args.no_configs:
        for cname in EXTRA:
            steps = max(3, args.steps // 4) if cname == "mixed" else args.steps
            extra[cname] = measure(cname, steps, args.warmup, world, rank, stream, peak, l2, flush)
            extra[cname]["workload"] = DESCRIPTIONS[cname]
            if rank == 0 and world == 1:
                extra[cname]["cpu_baseline"] = cpu_baselines(cname, rank, args.cpu_seconds)

    if not args.no_configs and world == 1:
        extra["indexer_logits"] = measure_logits(args.steps, args.warmup, stream, flush)
        if rank == 0:
            extra["indexer_logits"]["cpu_baseline"] = logits_cpu_baseline(args.cpu_seconds)

    if rank == 0:
        achieved = head["gbs_transform"]
        line = {
            "metric": METRIC,
            "value": head["rows_per_s"],
            "unit": "rows/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": head["us_per_step"] / 1e3,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded torch generators)",
            "config": headline_config(world, head["l2"]),
            "hbm_gbs": achieved,
            "hbm_frac_of_nominal_8tbs": head["frac_of_nominal_8tbs"],
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": profiled_traffic("topk_rows_kernel", "ragged_extend_chunk"),
                         "traffic_scope": "one 1024-row launch (ncu), per launch",
                         "kernel": "topk_rows_kernel<ragged> (transform launches in a CUDA graph, CUDA events)",
                         "alg_bytes_per_launch": head["alg_bytes_per_step"] // 16,
                         "us_per_launch": head["us_transform_per_step"] / 16},
            "gpu_launches": head["launches_per_step"] * args.steps,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": base,
            "configs": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
