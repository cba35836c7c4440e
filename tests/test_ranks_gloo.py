"""Multi-rank host logic of bench.py on CPU: two gloo ranks (127.0.0.1), each a
full replica of the workload (weak scaling, no data-path collective); the step
time is the maximum over ranks and the job rate counts every rank's units."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        lengths = bench.shard_sequences([8192] * 16, r, w)
        # rank 1 is the slow one in the first column, rank 0 in the second
        times = bench.max_over_ranks([5.0 + 2.0 * r, 3.0 - r, 1.0], dist)
        value = bench.job_throughput(w, bench.metric_flops(lengths, 12, 64), times[0])
        q.put((r, w, local, len(lengths), times, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicate_and_take_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    flops = bench.metric_flops([8192] * 16, 12, 64)
    for r, (rank, world, local, nseq, times, value) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert nseq == 16                       # every rank holds the whole workload
        assert times == [7.0, 3.0, 1.0]         # element-wise maximum over ranks
        assert value == pytest.approx(2 * flops / 7e-3)


def test_single_rank_identity():
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.job_throughput(1, 1e12, 1000.0) == pytest.approx(1e12)
