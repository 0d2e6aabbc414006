"""Two CPU ranks over gloo exercise the benchmark's multi-rank host logic:
the barrier, the max-over-ranks time, and the per-rank (weak-scaling)
workloads, which must differ between ranks while each rank's oracle result
stays its own. No GPU is used."""

from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        bench.barrier(world)
        t = bench.max_over_ranks(1.0 + rank, world)
        w = bench.make_workload("ragged_tiny", "cpu", rank)[0]
        out, _, _ = oracle.run_workload(w)
        digest = torch.tensor([int(out.astype("int64").sum() % (1 << 31))], dtype=torch.int64)
        gathered = [torch.zeros_like(digest) for _ in range(world)]
        dist.all_gather(gathered, digest)
        q.put((rank, t, [int(g) for g in gathered], int(w["seq_lens"].sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    assert all(t == 2.0 for _, t, _, _ in results)          # max over ranks
    assert results[0][2] == results[1][2]                    # all_gather agrees
    assert results[0][3] != results[1][3]                    # each rank has its own batch
