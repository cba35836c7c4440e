"""Host-side helpers of bench.py (no GPU): the work counts the throughput
lines divide by, and the CPU-affinity helper's parsing and fallback."""

import os

import bench
from oracle import backward_metric_flops, metric_flops


def test_forward_metric_counts_eight_n2d_per_head():
    assert bench.metric_flops([8192] * 16, 12, 64) == 8.0 * 8192 ** 2 * 64 * 12 * 16
    assert bench.metric_flops([3, 0, 5], 2, 32) == metric_flops([3, 0, 5], 2, 32)


def test_backward_counts():
    lengths, H, d, span = [100, 37], 3, 64, 256
    assert backward_metric_flops(lengths, H, d) == sum(22.0 * n * n * d * H for n in lengths)
    q, k = bench.bwd_kernel_flops(lengths, H, d, span)
    # the query kernel redoes the forward (two n^2 d products) on top of the key kernel's share
    n2 = sum(n * n for n in lengths) * d * H
    assert q - k == 2.0 * n2 + 8.0 * sum(lengths) * span * d * H


def test_cpulist_parsing():
    assert bench._cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench._cpulist("5") == {5}
    assert bench._cpulist("") == set()


def test_gpu_local_cpus_leaves_affinity_alone_without_a_device():
    before = os.sched_getaffinity(0)
    with bench.GpuLocalCpus(0) as numa:
        assert numa.node is None or isinstance(numa.node, int)
    assert os.sched_getaffinity(0) == before
