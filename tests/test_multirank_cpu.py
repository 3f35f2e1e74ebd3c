"""bench.py's multi-rank host logic on CPU ranks (gloo, world size 2): replicas
score their own seeded batches of one shape, the timed region is bracketed by
barriers, and the reported time is the maximum over ranks."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        spec = bench.replica_spec(workloads.WORKLOADS["tiny_bf16_1x4k"], rank, world)
        batch = workloads.make_batch(spec)
        bench.barrier(world)
        t = bench.max_over_ranks(1.5 + rank, world, "cpu")
        out[rank] = (spec.seed, tuple(batch.q.shape), float(batch.q.float().sum()), t)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    (s0, shape0, sum0, t0), (s1, shape1, sum1, t1) = out[0], out[1]
    assert shape0 == shape1            # same per-rank work (weak scaling)
    assert s0 != s1 and sum0 != sum1   # each replica draws its own inputs
    assert t0 == t1 == 2.5             # max over ranks, seen by every rank


def test_single_rank_is_unchanged():
    import bench
    import workloads
    spec = workloads.WORKLOADS["bf16_16x131k"]
    assert bench.replica_spec(spec, 0, 1) is spec
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0
