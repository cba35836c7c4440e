"""Multi-rank host logic of bench.py on CPU: two gloo ranks (127.0.0.1).  The
job holds one workload per rank; its sequences are split across ranks by a
greedy n^2-cost balance (sequences are independent, so there is no data-path
collective); the step time is the maximum over ranks and the job rate counts
every rank's units."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from exact_attention_deberta_gb300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _varlen_lengths():
    # the packed varlen workload's 64 lengths, uniform in [64, 2048]
    return [int(n) for n in synth.draw_lengths(synth.WORKLOADS["packed_varlen_h12d64"],
                                               np.random.default_rng(3))]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        lengths = bench.shard_sequences(_varlen_lengths(), r, w)
        shard = bench.assign_sequences(_varlen_lengths(), w)[r]
        # rank 1 is the slow one in the first column, rank 0 in the second
        times = bench.max_over_ranks([5.0 + 2.0 * r, 3.0 - r, 1.0], dist)
        value = bench.job_throughput(w, bench.metric_flops(_varlen_lengths(), 12, 64), times[0])
        q.put((r, w, local, lengths, shard, times, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_sequences_and_take_max():
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
    full = _varlen_lengths()
    flops = bench.metric_flops(full, 12, 64)
    seen = []
    costs = []
    for r, (rank, world, local, lengths, shard, times, value) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert times == [7.0, 3.0, 1.0]         # element-wise maximum over ranks
        assert value == pytest.approx(2 * flops / 7e-3)
        assert lengths == [full[s] for _, s in shard]
        seen += shard
        costs.append(sum(float(n) ** 2 for n in lengths))
    # every (copy, sequence) of the two-workload job exactly once
    assert sorted(seen) == [(c, s) for c in range(2) for s in range(len(full))]
    assert max(costs) / min(costs) <= 1.1


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_split_covers_the_job_and_balances(world):
    full = _varlen_lengths()
    shards = bench.assign_sequences(full, world)
    flat = sorted(e for sh in shards for e in sh)
    assert flat == [(c, s) for c in range(world) for s in range(len(full))]
    costs = [sum(float(full[s]) ** 2 for _, s in sh) for sh in shards]
    assert max(costs) / min(costs) <= 1.1
    # equal lengths: every rank gets exactly one workload's sequences
    eq = bench.assign_sequences([8192] * 16, world)
    assert all(len(sh) == 16 for sh in eq)


def test_shard_inputs_gathers_the_rank_tokens():
    x = synth.custom_inputs(layout="packed", dtype="bf16", H=2, d=64, lengths=[5, 300, 17, 129])
    for r in range(2):
        y = bench.shard_inputs(x, r, 2)
        mine = [s for _, s in bench.assign_sequences(x.lengths, 2)[r]]
        cu = x.cu_seqlens.numpy()
        want = torch.cat([x.q[cu[s]:cu[s + 1]] for s in mine])
        assert torch.equal(y.q, want)
        assert list(y.lengths) == [int(x.lengths[s]) for s in mine]
        assert int(y.cu_seqlens[-1]) == y.q.shape[0]
    xp = synth.custom_inputs(layout="padded", dtype="fp16", H=2, d=64, lengths=[5, 30, 17], L=32)
    y = bench.shard_inputs(xp, 1, 2)
    mine = [s for _, s in bench.assign_sequences(xp.lengths, 2)[1]]
    assert torch.equal(y.key_mask, xp.key_mask[mine])


def test_single_rank_identity():
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.job_throughput(1, 1e12, 1000.0) == pytest.approx(1e12)
    x = synth.custom_inputs(layout="packed", dtype="bf16", H=1, d=64, lengths=[3, 4])
    assert bench.shard_inputs(x, 0, 1) is x
