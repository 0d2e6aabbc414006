#!/usr/bin/env python3
"""Benchmark of the indexer top-k + transform on GB300.

One step = the whole hot path on one batch: topk_plan + the transform
(route, 16-byte window loads, key map, 12- or 14-bit first-digit
histogram, radix refine, compaction, fused page-table / offset emit).

Default workload (the headline line): PAGED decode, 128 rows x 8192 fp32
scores, k = 2048, page_size 64, a random page permutation. Those inputs
(5.3 MB) fit in L2, so every step uses the next of enough rotating input sets
to span more than twice the L2. The other workloads (RAGGED tiny, RAGGED
prefill extend, PAGED long, packed PAGED, the mixed sweep) are measured
after it and reported under "configs" in the same line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU with
its own seed (weak scaling; rows are independent, so there is no data-path
collective); the barrier and the max-over-ranks time use torch.distributed.
``--impl reference`` times the CPU oracle, as it stands, on host cores:
W untimed steps, then K timed steps of the headline workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
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
HEADLINE = "paged_decode"
REF_BUDGET_S = 150.0     # the whole reference-arm run, warm-up included
KERNEL_SRC = os.path.join(ROOT, "sparse_attention_top_row_gb300", "csrc", "topk.cu")


# ----------------------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"rows_kernel_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_src or not m_tr or m_src.group(1) != kernel_source_hash():
        return None
    return int(m_tr.group(1))


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

def make_workload(name, device, rank=0):
    """The named workload as a list of launches (each a workload dict)."""
    if name == "paged_decode":
        return [wl.paged_decode(device, sub_id=rank)]
    if name == "ragged_tiny":
        return [wl.ragged_tiny(device, sub_id=rank)]
    if name == "ragged_extend":
        return [wl.ragged_extend(device, chunk=c) for c in range(16)]
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


def algorithmic_bytes(w, out_raw):
    """Scores read by non-trivial rows + indices written + distinct page-table
    entries read + 4 B per per-row array read."""
    k = int(w["k"])
    lens = w["seq_lens"].to(torch.int64).clamp(min=0)
    nontrivial = lens > k
    scores = int((4 * lens[nontrivial]).sum().item())
    out = 4 * k * int(w["batch"])
    packed = [w.get(key) for key in ("page_table_row_starts", "row_to_batch")]
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


class Launch:
    """Device buffers + workspace for one launch, and its step function."""

    def __init__(self, w, flags=0):
        self.w = w
        self.B, self.k = int(w["batch"]), int(w["k"])
        self.out = torch.empty((self.B, self.k), dtype=torch.int32, device=w["scores"].device)
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
        else:
            topk.topk_transform_ragged(w["scores"], w["score_stride"], w.get("row_starts"), w["seq_lens"],
                                       w["out_offsets"], self.k, self.ws, self.out, out_raw, self.flags,
                                       stream=stream)

    def launches_per_step(self):
        return 2 + (1 if self.B <= 64 else 0)


def time_workload(launch_sets, steps, warmup, world, stream):
    """Times `steps` steps; timed step i runs every launch of set
    (warmup + i) % len(sets). The steps are captured into one CUDA graph (the
    way a serving loop launches them), so the device timeline holds no host
    launch gaps; a second graph of the transforms alone gives the per-launch
    duration of the transform. Returns (seconds for all steps, seconds per
    transform launch)."""
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
    # transforms alone (untimed for the headline value)
    ev[2].record(stream)
    g_tr.replay()
    ev[3].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev[0].record(stream)
    g_steps.replay()
    ev[1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total = ev[0].elapsed_time(ev[1]) / 1e3
    per_transform = ev[2].elapsed_time(ev[3]) / 1e3 / (steps * n_launch)
    del g_steps, g_tr
    return total, per_transform


def rotating_sets(name, device, rank, max_sets, flags=0):
    """Copies of a workload so that the timed steps never re-read a set that
    may still sit in L2: either one set already spans > 2x L2, or every step
    (warm-up and timed) gets a set of its own, up to `max_sets`."""
    base = make_workload(name, device, rank)
    size = sum(w["scores"].numel() * 4 for w in base)
    n = 1 if size > 2 * L2_BYTES else min(max_sets, int(math.ceil(2 * L2_BYTES / max(size, 1))) + 1)
    sets = [[Launch(w, flags) for w in base]]
    for c in range(1, n):
        sets.append([Launch({kk: (v.clone() if isinstance(v, torch.Tensor) else v) for kk, v in w.items()},
                            flags) for w in base])
    return sets, n


def measure(name, steps, warmup, world, rank, stream, peak):
    sets, n_sets = rotating_sets(name, "cuda", rank, max_sets=steps + warmup)
    # algorithmic bytes, from one run with out_raw
    alg = 0
    for ln in sets[0]:
        raw = torch.empty_like(ln.out)
        ln.plan(stream)
        ln.transform(stream, out_raw=raw)
        torch.cuda.synchronize()
        alg += algorithmic_bytes(ln.w, raw)
    rows = sum(ln.B for ln in sets[0])
    total, t_launch = time_workload(sets, steps, warmup, world, stream)
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
        "launches_per_step": sum(ln.launches_per_step() for ln in sets[0]),
        "rows_per_step": rows,
    }
    del sets
    torch.cuda.empty_cache()
    return res


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


def measure_e2e(name, steps, warmup, rank, stream):
    """Same metric through the public API with HOST buffers: each step copies
    the inputs from pinned host memory (all of a launch's inputs in one packed
    copy), plans, transforms and reads the output back to pinned host memory."""
    hosts = make_workload(name, "cpu", rank)
    packs = [packed_inputs(w, "cuda") for w in hosts]
    h2d = sum(hb.numel() for hb, _, _ in packs)
    d2h = sum(4 * int(w["batch"]) * int(w["k"]) for w in hosts)
    launches = [Launch(dw) for _, _, dw in packs]
    outs = [torch.empty((ln.B, ln.k), dtype=torch.int32).pin_memory() for ln in launches]

    def step():
        for (hb, db, _), ln, ho in zip(packs, launches, outs):
            db.copy_(hb, non_blocking=True)
            ln.plan(stream)
            ln.transform(stream)
            ho.copy_(ln.out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
    t = a.elapsed_time(b) / 1e3
    # One more step, untimed and in deterministic mode (a unique result), read
    # back to the host, must match a run on inputs copied the ordinary way
    # (sorted rows: the slot order is unspecified).
    for ln in launches:
        ln.flags = topk.TOPK_DETERMINISTIC
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    for w, ho in zip(hosts, outs):
        ref = Launch(wl.to_device(w, "cuda"), flags=topk.TOPK_DETERMINISTIC)
        ref.plan(stream)
        ref.transform(stream)
        torch.cuda.synchronize()
        if not torch.equal(torch.sort(ho, dim=1).values, torch.sort(ref.out.cpu(), dim=1).values):
            raise RuntimeError("end-to-end outputs differ from the device-resident run")
    rows = sum(ln.B for ln in launches)
    return {"value": rows * steps / t, "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


def cpu_baseline(name, budget_s, rank):
    """The CPU oracle, as it stands (single-threaded), on a bounded sample of
    the workload: whole launches repeated, or a prefix of rows for the big
    ones, until about `budget_s` seconds of CPU work."""
    import oracle
    launches = make_workload(name, "cpu", rank) if name not in ("ragged_extend",) else \
        [wl.ragged_extend("cpu", chunk=0, rows_per_chunk=64)]
    rows_done, t0 = 0, time.perf_counter()
    reps = 0
    while time.perf_counter() - t0 < budget_s:
        for w in launches:
            oracle.run_workload(w)
            rows_done += int(w["batch"])
        reps += 1
    t = time.perf_counter() - t0
    sample = (f"{reps} pass(es) over {'the first 64 rows of chunk 0' if name == 'ragged_extend' else 'the whole batch'}"
              f" of the {name} workload ({rows_done} rows)")
    return {"value": rows_done / t, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": sample}


# ----------------------------------------------------------------------------- main

def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands (single-threaded), on
    the headline workload. W untimed steps, then exactly K timed steps; a step
    is the oracle over the whole batch, or over its first R rows when K + W
    whole batches would take longer than REF_BUDGET_S (R is chosen from the
    time of the first warm-up step). Rank 0 alone runs it."""
    if rank != 0:
        return
    import oracle
    w = make_workload(HEADLINE, "cpu", rank)[0]
    B = int(w["batch"])
    t0 = time.perf_counter()
    oracle.run_workload(w)                      # the first warm-up step
    t_batch = time.perf_counter() - t0
    n_steps = args.steps + args.warmup
    rows_per_step = B
    if t_batch * n_steps > REF_BUDGET_S:
        rows_per_step = max(1, int(B * REF_BUDGET_S / (t_batch * n_steps)))
    rows = None if rows_per_step == B else list(range(rows_per_step))
    for _ in range(args.warmup - 1):
        oracle.run_workload(w, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run_workload(w, rows=rows)
    t = time.perf_counter() - t0
    value = rows_per_step * args.steps / t
    what = "the whole batch" if rows is None else f"the first {rows_per_step} of its {B} rows"
    base = {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": f"{args.steps} timed step(s) after {args.warmup} warm-up step(s), each the oracle over "
                      f"{what} of the {HEADLINE} workload"}
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)", "impl": "reference",
        "config": {"workload": "PAGED decode B=128 L=8192 k=2048 page_size=64",
                   "global_batch": 128, "seq_len": 8192, "parallelism": f"rows x{args.gpus} (weak)"},
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-configs", action="store_true", help="headline workload only")
    ap.add_argument("--workload", default=HEADLINE, help="headline workload (default: paged_decode)")
    ap.add_argument("--quick", action="store_true",
                    help="the headline workload only: no other configs, no e2e, no CPU baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
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

    with ClockSampler(local) as clocks:
        head = measure(args.workload, args.steps, args.warmup, world, rank, stream, peak)
    clk = clocks.summary()
    if args.quick:
        if rank == 0:
            print(json.dumps({"workload": args.workload, **head, "clocks": clk}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    extra = {}
    if not args.no_configs:
        for name, steps in (("ragged_tiny", args.steps), ("ragged_extend", max(3, args.steps // 10)),
                            ("paged_long_b1", args.steps), ("paged_long_b30", args.steps),
                            ("paged_long_b31", args.steps), ("paged_packed", args.steps),
                            ("mixed", max(3, args.steps // 10))):
            extra[name] = measure(name, steps, args.warmup if name != "ragged_extend" else 3,
                                  world, rank, stream, peak)

    e2e = measure_e2e(HEADLINE, args.steps, args.warmup, rank, stream)
    base = cpu_baseline(HEADLINE, args.cpu_seconds, rank) if (rank == 0 and world == 1) else None

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
            "config": {"workload": "PAGED decode B=128 L=8192 k=2048 page_size=64 (random page permutation)",
                       "global_batch": 128 * world, "seq_len": 8192, "k": 2048,
                       "parallelism": f"rows x{world} (weak)",
                       "l2": f"{head['input_sets']} rotating input sets (> 2x L2 per cycle)"},
            "hbm_gbs": achieved,
            "hbm_frac_of_nominal_8tbs": head["frac_of_nominal_8tbs"],
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": profiled_traffic(HEADLINE),
                         "kernel": "topk_rows_kernel<paged> (transform launches in a CUDA graph, CUDA events)",
                         "alg_bytes_per_launch": head["alg_bytes_per_step"]},
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
