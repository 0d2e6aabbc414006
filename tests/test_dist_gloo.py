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


def _partition_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from sparse_attention_top_row_gb300 import workloads as wl
        results = {}
        for name, w in (("ragged", wl.mixed("cpu", mode="ragged", k=256, batch=13, max_len=20000, sub_id=5)),
                        ("paged", wl.mixed("cpu", mode="paged", k=512, batch=13, max_len=20000, sub_id=6)),
                        ("packed", wl.paged_packed("cpu", n_req=3, q_rows=3, min_tokens=3000, max_tokens=6000,
                                                   window=4000, k=300))):
            shard = wl.shard_rows(w, rank, world)
            out = oracle.run_workload(shard)[0] if shard is not None else None
            gathered = [None] * world
            dist.all_gather_object(gathered, out)          # the one exchange: outputs to every rank
            results[name] = [g for g in gathered if g is not None]
        q.put((rank, results))
    finally:
        dist.destroy_process_group()


def test_rows_partitioned_over_two_gloo_ranks():
    """One batch's rows split contiguously over two ranks, each shard run
    through the oracle, the outputs gathered: the concatenation equals the
    one-rank result on the whole batch (plain RAGGED and PAGED rows, and
    packed PAGED rows, whose shards keep the request tables)."""
    import numpy as np

    import oracle
    from sparse_attention_top_row_gb300 import workloads as wl
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_partition_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    whole = {"ragged": wl.mixed("cpu", mode="ragged", k=256, batch=13, max_len=20000, sub_id=5),
             "paged": wl.mixed("cpu", mode="paged", k=512, batch=13, max_len=20000, sub_id=6),
             "packed": wl.paged_packed("cpu", n_req=3, q_rows=3, min_tokens=3000, max_tokens=6000, window=4000,
                                       k=300)}
    for name, w in whole.items():
        ref = oracle.run_workload(w)[0]
        for rank in (0, 1):
            got = np.concatenate(results[rank][name])
            np.testing.assert_array_equal(got, ref, err_msg=name)


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
