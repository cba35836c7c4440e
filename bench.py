"""Throughput of the fused disentangled-attention forward on GB300.

One step = one df_attn_fwd call (planning kernel + fused attention kernels)
over the long-context packed workload: 16 sequences of 8192 tokens, H = 12,
d = 64, bf16 (DeBERTa-v3-base heads), inputs resident in HBM.  The metric is
TFLOP/s counted as 8 n^2 d per head over valid tokens, plus tokens/s and the
fraction of the dense bf16 tensor peak.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

With N > 1 (torchrun, one rank per GPU) every rank runs its own copy of the
workload (independent sequences, no collective on the data path): weak scaling.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

DEFAULT_WORKLOAD = "long_packed_h12d64"
L2_BYTES = 129e6  # GB300 L2 cache
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fp32-mode", choices=["strict", "fast"], default="strict",
                    help="fp32 workloads: the strict CUDA-core kernel, or the fast mode "
                         "(df_attn_fwd_fp32_fast: fp16 tensor-core path, no host-buffer e2e)")
    ap.add_argument("--group-tokens", type=int, default=0,
                    help="host-buffer forward: tokens per group of sequences (0: B*L/4)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--small-calls", type=int, default=200,
                    help="--op small: timed calls per workload and mode (a few for a profiler's launch list)")
    ap.add_argument("--op", choices=["attention", "pack", "linear", "encoder", "bwd", "small"], default="attention",
                    help="pack: the padded <-> packed conversion; linear: the QKV and PK/PQ projections; "
                         "encoder: a 12-layer DeBERTa-v3-base encoder on synthetic weights; "
                         "bwd: the backward pass (dQ, dK, dV, dPK, dPQ) of the attention; "
                         "small: per-call latency of the small padded workloads (launch / HBM bound)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def assign_sequences(lengths, world: int):
    """Split of the job's sequences across ranks (weak scaling: the job holds
    `world` copies of the workload's sequence set, so a rank's share is one
    workload's worth of work).  Sequences are independent (the DisentangledFlash
    discussion's packed-vs-padded paragraph: each sequence is its own problem, no
    computation crosses a boundary), so no collective is needed on the data path.
    Greedy longest-processing-time balance on the n^2 cost: sequences in
    non-increasing length order, each to the rank with the least cost so far
    (ties: lowest rank).  Returns, per rank, a list of (copy, sequence index)."""
    job = [(c, s, int(n)) for c in range(world) for s, n in enumerate(lengths)]
    job.sort(key=lambda e: -e[2])  # stable: equal lengths keep (copy, index) order
    load = [0.0] * world
    shards = [[] for _ in range(world)]
    for c, s, n in job:
        r = min(range(world), key=lambda i: (load[i], i))
        shards[r].append((c, s))
        load[r] += float(n) * float(n)
    for sh in shards:
        sh.sort()
    return shards


def shard_sequences(lengths, rank: int, world: int):
    """Lengths of the sequences rank `rank` processes (see assign_sequences)."""
    return [int(lengths[s]) for _, s in assign_sequences(lengths, world)[rank]]


def shard_inputs(x, rank: int, world: int):
    """This rank's inputs: the tokens (packed) or batch rows (padded) of its
    sequences, gathered on the host into a new contiguous batch."""
    mine = [s for _, s in assign_sequences(x.lengths, world)[rank]]
    if world == 1:
        return x
    import dataclasses
    if x.w.layout == "packed":
        cu = x.cu_seqlens.numpy()
        idx = torch.cat([torch.arange(int(cu[s]), int(cu[s + 1])) for s in mine]) if mine else \
            torch.zeros(0, dtype=torch.long)
        n = np.asarray([int(x.lengths[s]) for s in mine], dtype=np.int64)
        cuv = torch.zeros(n.size + 1, dtype=torch.int32)
        cuv[1:] = torch.from_numpy(np.cumsum(n).astype(np.int32))
        return dataclasses.replace(x, lengths=n, q=x.q[idx].contiguous(), k=x.k[idx].contiguous(),
                                   v=x.v[idx].contiguous(), cu_seqlens=cuv)
    rows = torch.tensor(mine, dtype=torch.long)
    return dataclasses.replace(x, lengths=np.asarray([int(x.lengths[s]) for s in mine], dtype=np.int64),
                               q=x.q[rows].contiguous(), k=x.k[rows].contiguous(),
                               v=x.v[rows].contiguous(), key_mask=x.key_mask[rows].contiguous())


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of per-rank timings (the slowest rank decides the
    step time); identity with one rank."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_throughput(world: int, units_per_rank: float, ms: float) -> float:
    """Whole-job rate: the units all ranks processed in one step (each rank
    holds one workload's worth, `world` workloads in all) over the step time,
    the maximum over ranks."""
    return world * units_per_rank / (ms * 1e-3)


def metric_flops(lengths, H, d):
    return float(sum(8.0 * n * n * d * H for n in lengths))


def algorithmic_flops(lengths, H, d, span):
    """Dense contractions the method needs: Q.K^T and P.V (2 n^2 d each) plus the
    two relative-position projections Q.PK^T and K.PQ^T (2 n (2 span) d each)."""
    return float(sum(H * (4.0 * n * n * d + 8.0 * n * span * d) for n in lengths))


def tile_flops(lengths, H, d, span, rsp, rsn):
    """Algorithmic flops per launch of the near-tile and far-tile kernels: Q.K^T and
    P.V over the valid (query, key) pairs of every 128 x 128 tile (4 rows keys d),
    split by the tile's class (far: every distance saturated, r - 127 >= r_sat_pos
    or r + 127 <= r_sat_neg for the tile offset r); the two relative-position
    projections (8 n span d per sequence and head) belong to the near-tile kernel."""
    near = far = 0.0
    for n in lengths:
        nb = (n + 127) // 128
        rows = [min(128, n - 128 * b) for b in range(nb)]
        for ib in range(nb):
            for jb in range(nb):
                off = 128 * (ib - jb)
                f = 4.0 * rows[ib] * rows[jb] * d
                if off - 127 >= rsp or off + 127 <= rsn:
                    far += f
                else:
                    near += f
        near += 8.0 * n * span * d
    return H * near, H * far


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(PEAKS_FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [c.strip() for c in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def _cpulist(text: str):
    cpus = set()
    for part in text.strip().split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus


class GpuLocalCpus:
    """Runs the process on the CPUs of the GPU's NUMA node while page-locked
    host buffers are allocated and used, so that they sit in the memory the
    GPU reaches without crossing to another socket (sysfs: the GPU's PCI
    function and its node's cpulist); the previous affinity comes back on
    exit.  `node` is None where the topology cannot be read."""

    def __init__(self, device: int):
        self.device = device
        self.node = None
        self.saved = None

    def __enter__(self):
        try:
            p = torch.cuda.get_device_properties(self.device)
            bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
            with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
                node = int(f.read())
            if node >= 0:
                with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
                    cpus = _cpulist(f.read()) & os.sched_getaffinity(0)
                if cpus:
                    self.saved = os.sched_getaffinity(0)
                    os.sched_setaffinity(0, cpus)
                    self.node = node
        except Exception:  # no device, no sysfs entry, an unreadable topology: leave affinity alone
            self.node = None
        return self

    def __exit__(self, *exc):
        if self.saved is not None:
            os.sched_setaffinity(0, self.saved)


def traffic_record(kernel_file: str, workload: str):
    """DRAM bytes per launch of the dominant kernel on this workload from the
    committed ncu summary (entries keyed "<source file>@<workload>"), valid only
    while the kernel source is unchanged since the capture."""
    rec = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "exact_attention_deberta_gb300", "csrc", kernel_file)
    if not (os.path.exists(rec) and os.path.exists(src)):
        return None
    with open(rec) as f:
        data = json.load(f)
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    entry = data.get(f"{kernel_file}@{workload}")
    if not entry or entry.get("source_sha256_16") != digest or entry.get("workload") != workload:
        return None
    return entry


def cpu_oracle_rate(x, budget_s: float = 12.0):
    """The float64 oracle, as it stands, on a bounded sample of the same workload:
    query rows of the first sequence / head.  Returns (TFLOP/s-equivalent, tokens/s,
    rows, seconds, threads)."""
    from oracle import attend_rows
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    st, n = x.seq_slices()[0]
    sl = lambda t: t[st:st + n] if x.w.layout == "packed" else t[0, :n]  # noqa: E731
    q, k, v = sl(x.q), sl(x.k), sl(x.v)
    rows_done, t_used, m = 0, 0.0, 32
    while t_used < budget_s:
        rows = np.arange(m) % n
        t0 = time.perf_counter()
        attend_rows(q, k, v, x.pk, x.pq, 0, rows, **kw)
        dt = time.perf_counter() - t0
        rows_done += m
        t_used += dt
        if dt < budget_s / 8:
            m *= 2
    flops = rows_done * 8.0 * n * x.w.d        # per row: 8 n d of the metric's 8 n^2 d
    threads = _blas_threads()
    return flops / t_used / 1e12, rows_done / t_used, rows_done, t_used, threads


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return int(max(i.get("num_threads", 1) for i in info))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, rank, world):
    """Reference arm: the float64 oracle timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    from exact_attention_deberta_gb300 import synth
    x = synth.make_inputs(args.workload)
    from oracle import attend_rows
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    st, n = x.seq_slices()[0]
    sl = lambda t: t[st:st + n] if x.w.layout == "packed" else t[0, :n]  # noqa: E731
    q, k, v = sl(x.q), sl(x.k), sl(x.v)
    rows = np.arange(64)
    for _ in range(args.warmup):
        attend_rows(q, k, v, x.pk, x.pq, 0, rows[:8], **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        attend_rows(q, k, v, x.pk, x.pq, 0, rows, **kw)
    dt = time.perf_counter() - t0
    flops = args.steps * rows.size * 8.0 * n * x.w.d
    value = flops / dt / 1e12
    cores = _blas_threads()
    sample = f"{rows.size} query rows x 1 head of one {n}-token sequence per step"
    line = {"impl": "reference", "metric": "disentangled-attn fwd TFLOP/s (8*L^2*d/head)",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": x.w.name, "sequences": len(x.lengths), "seq_len": int(x.w.L),
                       "H": x.w.H, "d": x.w.d, "io_dtype": x.w.dtype, "layout": x.w.layout,
                       "buckets": x.w.buckets, "max_rel": x.w.max_rel, "span": x.w.span},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_pack(args, local):
    """Padded <-> packed conversion (HBM-bound row gathers): GB/s of df_pack_rows
    and df_unpack_rows on right-padded batches, against the measured HBM copy
    rate, with the mask metadata (df_pack_info) timed beside them."""
    torch.cuda.set_device(local)
    from exact_attention_deberta_gb300.build import build
    build()
    from exact_attention_deberta_gb300 import binding
    peaks, src = load_peaks()
    rng = np.random.default_rng(4)
    shapes = {
        # 16 x 8192 right-padded, lengths U{2048..8192}, hidden 768 bf16 (q of the long workload)
        "long_padded_b16_l8192_h768_bf16": (16, 8192, 768, torch.bfloat16,
                                            rng.integers(2048, 8193, 16)),
        # MNLI-like padding (lognormal lengths, 93 % padding), hidden 24 x 64 fp16
        "mnli_like_b16_l512_h1536_fp16": (16, 512, 1536, torch.float16,
                                          np.clip(np.round(np.random.default_rng(2).lognormal(np.log(30), 0.65, 16)),
                                                  8, 512).astype(np.int64)),
    }
    stream = torch.cuda.current_stream()
    out_lines = {}
    for name, (B, L, D, dt, lengths) in shapes.items():
        mask = torch.from_numpy((np.arange(L)[None, :] < lengths[:, None]).astype(np.uint8)).cuda()
        x = torch.randn(B, L, D, device="cuda").to(dt)
        info = binding.df_pack_info(mask)
        T, row = info.total, D * x.element_size()
        tokens = torch.empty(max(T, 1), D, dtype=dt, device="cuda")
        out = torch.empty_like(x)
        lib = binding.raw_library
        sp = binding._stream(stream)

        def pack():
            return lib.df_pack_rows(binding._ptr(x), binding._ptr(info.indices), binding._ptr(info.stats),
                                    B * L, row, binding._ptr(tokens), sp)

        def unpack():
            return lib.df_unpack_rows(binding._ptr(tokens), binding._ptr(info.inverse), B * L, row,
                                      binding._ptr(out), sp)

        def meta():
            return lib.df_pack_info(binding._ptr(mask), B, L, binding._ptr(info.cu_seqlens),
                                    binding._ptr(info.indices), binding._ptr(info.inverse),
                                    binding._ptr(info.stats), sp)

        res = {}
        for op, fn, nbytes in (("pack", pack, 2 * T * row + 4 * T),
                               ("unpack", unpack, B * L * row + T * row + 4 * B * L),
                               ("info", meta, B * L + 4 * (2 * B * L + B + 3))):
            for _ in range(args.warmup):
                assert fn() == binding.DF_OK
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            res[op] = {"ms": ms, "bytes": int(nbytes), "gbs": nbytes / ms / 1e6}
        # the oracle on the host, same rows
        t0 = time.perf_counter()
        from oracle import pack_info as o_info, pack_rows as o_pack, unpack_rows as o_unpack
        xm = x.view(torch.uint8).cpu().numpy().reshape(B * L, -1)
        _, idx, inv, _, _ = o_info(mask.cpu().numpy())
        tok = o_pack(xm, idx)
        o_unpack(tok, inv)
        cpu_s = time.perf_counter() - t0
        out_lines[name] = {"tokens": T, "row_bytes": row, **res,
                           "cpu_baseline": {"value": (res["pack"]["bytes"] + res["unpack"]["bytes"]) / cpu_s / 1e9,
                                            "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                                            "sample": "whole workload: metadata, pack and unpack, numpy"}}
    head = out_lines["long_padded_b16_l8192_h768_bf16"]
    gbs = (head["pack"]["bytes"] + head["unpack"]["bytes"]) / (head["pack"]["ms"] + head["unpack"]["ms"]) / 1e6
    line = {"metric": "padded<->packed conversion GB/s (pack + unpack bytes)", "value": gbs, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "bytes", "data": "synthetic",
            "config": {"workload": "long_padded_b16_l8192_h768_bf16",
                       "l2": "inputs larger than L2 (x 201 MB, out 201 MB)"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None, "peak_source": src + " hbm_gbs"},
            "workloads": out_lines, "gpu_launches": 2 * args.steps}
    print(json.dumps(line), flush=True)


def run_linear(args, local):
    """The projections that feed the attention (df_linear): the fused QKV
    projection of the 16 x 8192-token workload (hidden 768 -> 3 x 768, bf16) and
    the PK/PQ projection of 512 relative embeddings, as TFLOP/s against the
    measured dense bf16 rate (the kernel is timed alone: burst figure)."""
    torch.cuda.set_device(local)
    from exact_attention_deberta_gb300.build import build
    build()
    from exact_attention_deberta_gb300 import binding
    peaks, src = load_peaks()
    g = torch.Generator().manual_seed(4)
    res = {}
    for name, (M, K, N, n_out) in {"qkv_t131072_h768_bf16": (131072, 768, 768, 3),
                                   "pkpq_r512_h768_bf16": (512, 768, 768, 2)}.items():
        x = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
        ws = [(torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16).cuda() for _ in range(n_out)]
        bs = [(torch.randn(N, generator=g) * 0.1).to(torch.bfloat16).cuda() for _ in range(n_out)]
        outs = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(n_out)]
        for _ in range(args.warmup):
            binding.df_linear(x, ws, bs, outs)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            binding.df_linear(x, ws, bs, outs)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        flops = 2.0 * M * K * N * n_out
        res[name] = {"ms": ms, "flops": flops, "tflops": flops / ms / 1e9,
                     "bytes": 2 * (M * K + n_out * (N * K + N + M * N))}
    # the oracle (numpy float64 matmul) on a 1024-row sample of the QKV case
    from oracle import linear as o_linear
    xs = np.random.default_rng(0).standard_normal((1024, 768))
    wn = [np.random.default_rng(i).standard_normal((768, 768)) for i in range(3)]
    t0 = time.perf_counter()
    o_linear(xs, wn)
    cpu = 2.0 * 1024 * 768 * 768 * 3 / (time.perf_counter() - t0) / 1e12
    head = res["qkv_t131072_h768_bf16"]
    line = {"metric": "QKV projection TFLOP/s (2 M K N per output)", "value": head["tflops"], "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms"],
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "qkv_t131072_h768_bf16", "l2": "x 201 MB, outputs 604 MB: larger than L2"},
            "roofline": {"bound": "tensor", "achieved": head["tflops"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": head["tflops"] / peaks["bf16_tflops"], "traffic": None,
                         "peak_source": src + " bf16_tflops (burst)"},
            "workloads": res, "gpu_launches": args.steps,
            "cpu_baseline": {"value": cpu, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": "1024 x 768 rows by three 768 x 768 weights, float64 numpy"}}
    print(json.dumps(line), flush=True)


def run_small(args, local):
    """The small workloads, where launch latency and HBM set the time: per call,
    >= 200 back-to-back calls timed one by one with CUDA events (median and
    mean), both as eager calls and as the replay of a CUDA graph that holds one
    call; TFLOP/s on the metric's count and GB/s of algorithmic bytes (Q, K, V,
    O of the valid tokens, PK and PQ, the mask) against the measured HBM rate.
    The float64 oracle is timed on each workload in full."""
    torch.cuda.set_device(local)
    from exact_attention_deberta_gb300.build import build
    build()
    from exact_attention_deberta_gb300 import binding, synth
    from oracle import attend_padded
    peaks, src = load_peaks()
    calls = max(1, args.small_calls)
    stream = torch.cuda.current_stream()
    res = {}
    for name in ("tiny_fp32", "tiny_fp32_pad97", "v3base_padded_bf16", "v2xl_heavypad_fp16"):
        x = synth.make_inputs(name)
        H, d, span, L = x.w.H, x.w.d, x.w.span, x.w.L
        kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=span)
        dev = {n: getattr(x, n).cuda() for n in ("q", "k", "v", "pk", "pq", "key_mask")}
        out = torch.empty_like(dev["q"])
        B = dev["q"].shape[0]
        ws = torch.empty(binding.df_attn_workspace_size(B, H, L, d, **kw), dtype=torch.uint8, device="cuda")

        def call():
            binding.df_attn_fwd(dev["q"], dev["k"], dev["v"], dev["pk"], dev["pq"], key_mask=dev["key_mask"],
                                out=out, workspace=ws, **kw)

        for _ in range(max(3, args.warmup)):
            call()
        torch.cuda.synchronize()
        launches = binding.df_attn_last_launch_count()

        def timed(fn):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(calls + 1)]
            ev[0].record(stream)
            for i in range(calls):
                fn()
                ev[i + 1].record(stream)
            torch.cuda.synchronize()
            t = [ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(calls)]
            return float(np.median(t)), float(np.mean(t))

        eager = timed(call)
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                call()
            graph.replay()
            torch.cuda.synchronize()
            replay = timed(graph.replay)
        except RuntimeError as e:  # a capture the runtime refuses: report the eager calls only
            print(f"graph capture of {name} failed: {e}", file=sys.stderr)
            replay = eager
        assert binding.df_attn_get_device_status(ws) == binding.DF_OK
        lengths = [int(n) for n in x.lengths]
        flops = metric_flops(lengths, H, d)
        es = out.element_size()
        T = sum(lengths)
        nbytes = 4 * T * H * d * es + 2 * 2 * span * H * d * es + B * L
        oracle_s = None
        if not args.no_cpu_baseline:
            t0 = time.perf_counter()
            attend_padded(x.q, x.k, x.v, x.pk, x.pq, x.key_mask, **kw)
            oracle_s = time.perf_counter() - t0
        res[name] = {"tokens": T, "launches_per_call": launches, "flops": flops, "bytes": nbytes,
                     "eager_us_median": eager[0], "eager_us_mean": eager[1],
                     "graph_us_median": replay[0], "graph_us_mean": replay[1],
                     "tflops_graph": flops / (replay[0] * 1e-6) / 1e12,
                     "gbs_graph": nbytes / (replay[0] * 1e-6) / 1e9,
                     "hbm_frac_graph": nbytes / (replay[0] * 1e-6) / 1e9 / peaks["hbm_gbs"],
                     "oracle_s_full": oracle_s}
    head = res["v3base_padded_bf16"]
    line = {"metric": "small padded batch latency (us per call, CUDA-graph replay, median)",
            "value": head["graph_us_median"], "unit": "us", "n_gpus": 1, "steps": calls, "warmup": max(3, args.warmup),
            "ms_per_step": head["graph_us_median"] / 1e3, "higher_is_better": False, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "v3base_padded_bf16", "B": 16, "L": 512, "H": 12, "d": 64,
                       "l2": "inputs smaller than L2: back-to-back calls, as the workload's own use"},
            "roofline": {"bound": "hbm", "achieved": head["gbs_graph"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": head["hbm_frac_graph"], "traffic": None, "peak_source": src + " hbm_gbs"},
            "workloads": res, "gpu_launches": head["launches_per_call"] * calls * 2,
            "cpu_baseline": None if head["oracle_s_full"] is None else
            {"value": head["oracle_s_full"] * 1e6, "unit": "us", "cores": torch.get_num_threads(),
             "kind": "oracle", "sample": "each workload in full, float64 numpy"}}
    print(json.dumps(line), flush=True)


def bwd_kernel_flops(lengths, H, d, span):
    """Algorithmic flops of the two backward tile kernels.  Query kernel: the
    forward recomputed (Q.K^T and P.V) and a second Q.K^T with dP = dO.V^T and
    dQ = dS.K, 10 n^2 d; key kernel: Q.K^T, dP, dK = dS^T.Q and dV = P^T.dO,
    8 n^2 d.  Each recomputation of the scores also costs the two position
    projections, 8 n span d (two in the query kernel, one in the key kernel)."""
    q = sum(H * (10.0 * n * n * d + 16.0 * n * span * d) for n in lengths)
    k = sum(H * (8.0 * n * n * d + 8.0 * n * span * d) for n in lengths)
    return float(q), float(k)


def run_bwd(args, local):
    """Backward pass of the attention (df_attn_bwd, strict fp32 on CUDA cores)
    over the same workload as the forward bench; the metric counts 22 n^2 d per
    head (the eleven n x n x d products of the direct formulation)."""
    torch.cuda.set_device(local)
    from exact_attention_deberta_gb300.build import build
    build()
    from exact_attention_deberta_gb300 import binding, synth
    from oracle import backward_head, backward_metric_flops
    x = synth.make_inputs(args.workload)
    H, d, span = x.w.H, x.w.d, x.w.span
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=span)
    host = {n: getattr(x, n) for n in ("q", "k", "v", "pk", "pq", "key_mask", "cu_seqlens")
            if getattr(x, n) is not None}
    host["dout"] = synth.grad_output(x)
    dev = {n: t.cuda() for n, t in host.items()}
    B = len(x.lengths)
    ws = torch.empty(binding.df_attn_bwd_workspace_size(B, H, x.w.L, d, **kw), dtype=torch.uint8,
                     device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    grads = tuple(torch.empty(dev["q"].shape, **f32) for _ in range(3)) + tuple(
        torch.empty(dev["pk"].shape, **f32) for _ in range(2))
    stream = torch.cuda.current_stream()

    def step(inp):
        mode = (dict(cu_seqlens=inp["cu_seqlens"], max_seqlen=x.w.L) if x.w.layout == "packed"
                else dict(key_mask=inp["key_mask"]))
        binding.df_attn_bwd(inp["q"], inp["k"], inp["v"], inp["pk"], inp["pq"], inp["dout"], grads=grads,
                            workspace=ws, **mode, **kw)

    for _ in range(args.warmup):
        step(dev)
    torch.cuda.synchronize()
    assert binding.df_attn_get_device_status(ws) == binding.DF_OK
    launches = binding.df_attn_last_launch_count()
    kev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    for evs in kev:
        for e in evs:
            e.record(stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0.record(stream)
        for i in range(args.steps):
            binding.df_attn_set_profile_events(kev[i][0], kev[i][2])
            binding.df_attn_set_profile_split(kev[i][1])
            step(dev)
        t1.record(stream)
        torch.cuda.synchronize()
    binding.df_attn_set_profile_events(None, None)
    binding.df_attn_set_profile_split(None)
    ms = t0.elapsed_time(t1) / args.steps
    q_ms = sum(a.elapsed_time(m) for a, m, _ in kev) / args.steps
    k_ms = sum(m.elapsed_time(b) for _, m, b in kev) / args.steps
    e2e = None
    if not args.no_e2e:
        pinned = {n: t.pin_memory() for n, t in host.items()}
        dev2 = {n: torch.empty_like(t) for n, t in dev.items()}
        outs = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in grads]
        h2d = sum(t.numel() * t.element_size() for t in pinned.values())
        d2h = sum(t.numel() * t.element_size() for t in outs)
        steps_e2e = max(1, min(args.steps, 3))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps_e2e):
            for n in pinned:
                dev2[n].copy_(pinned[n], non_blocking=True)
            step(dev2)
            for o, g in zip(outs, grads):
                o.copy_(g, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e = (e0.elapsed_time(e1) / steps_e2e, h2d, d2h)
    flops = backward_metric_flops(x.lengths, H, d)
    value = flops / ms / 1e9
    q_flops, k_flops = bwd_kernel_flops(x.lengths, H, d, span)
    peak = 152 * 128 * 2 * 2.07e9 / 1e12
    kern = [("bwd_q_kernel", q_flops, q_ms), ("bwd_k_kernel", k_flops, k_ms)]
    kern.sort(key=lambda t: -t[2])
    (kname, kfl, kms), (oname, ofl, oms) = kern
    line = {"metric": "disentangled-attn bwd TFLOP/s (22*L^2*d/head)", "value": value, "unit": "TFLOP/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": x.w.name, "sequences": len(x.lengths), "seq_len": int(x.w.L), "H": H,
                       "d": d, "io_dtype": x.w.dtype, "grad_dtype": "fp32", "layout": x.w.layout,
                       "buckets": x.w.buckets, "max_rel": x.w.max_rel, "span": span,
                       "l2": "inputs and gradients larger than L2"},
            "gpu_launches": launches * args.steps,
            "roofline": {"bound": "alu", "achieved": kfl / (kms * 1e-3) / 1e12, "peak": peak, "unit": "TFLOP/s",
                         "frac": kfl / (kms * 1e-3) / 1e12 / peak, "traffic": None, "kernel": kname,
                         "kernel_ms": kms, "algorithmic_flops": kfl,
                         "peak_source": "derived: 152 SM x 128 FP32 lanes x 2 x 2.07 GHz",
                         "other_kernel": {"kernel": oname, "kernel_ms": oms, "algorithmic_flops": ofl,
                                          "achieved": ofl / (oms * 1e-3) / 1e12,
                                          "frac": ofl / (oms * 1e-3) / 1e12 / peak},
                         "rest_ms": ms - q_ms - k_ms},
            "clocks": clk.summary()}
    if e2e:
        line["e2e"] = {"value": flops / e2e[0] / 1e9, "unit": "TFLOP/s", "h2d_bytes_per_step": e2e[1],
                       "d2h_bytes_per_step": e2e[2]}
    if not args.no_cpu_baseline:
        # the first sequence, heads 0..2 (about 10 s of float64 work on 16 cores)
        n = int(x.lengths[0])
        st = int(x.cu_seqlens[0]) if x.w.layout == "packed" else 0
        sl = slice(st, st + n)
        heads = min(3, H)
        t_0 = time.perf_counter()
        for h in range(heads):
            a = [t[sl, h] for t in (x.q, x.k, x.v)] + [x.pk[:, h], x.pq[:, h], host["dout"][sl, h]]
            backward_head(*a, **kw)
        secs = time.perf_counter() - t_0
        line["cpu_baseline"] = {"value": heads * 22.0 * n * n * d / secs / 1e12, "unit": "TFLOP/s",
                                "cores": torch.get_num_threads(), "kind": "oracle",
                                "sample": f"backward of heads 0..{heads - 1} of one {n}-token sequence, "
                                          f"float64 numpy, {secs:.1f} s"}
    print(json.dumps(line), flush=True)


def run_encoder(args, local):
    """The pages' benchmark workload in kind: a 12-layer DeBERTa-v3-base encoder
    (hidden 768, 12 heads, FFN 3072, buckets 256, max_rel 512) on the packed
    layout with synthetic weights, packed lengths uniform in [0.6 L, L]
    (L = 8192), bf16; latency of one forward (mean over `steps` fresh inputs)."""
    torch.cuda.set_device(local)
    from exact_attention_deberta_gb300.build import build
    build()
    from exact_attention_deberta_gb300.encoder import Encoder, EncoderConfig, synthetic_weights
    cfg = EncoderConfig()
    layers, shared = synthetic_weights(cfg, seed=0)
    enc = Encoder(cfg, layers, shared)
    L = 8192
    rng = np.random.default_rng(0)
    res = {}
    for B in (1, 16):
        times, toks = [], []
        for it in range(args.warmup + args.steps):
            lengths = rng.integers(int(0.6 * L), L + 1, B)
            T = int(lengths.sum())
            cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device="cuda")
            h = torch.randn(T, cfg.hidden, device="cuda").to(torch.bfloat16)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            enc(h, cu, L)
            e1.record()
            torch.cuda.synchronize()
            if it >= args.warmup:
                times.append(e0.elapsed_time(e1))
                toks.append(T)
        ms = float(np.mean(times))
        res[f"b{B}_l{L}"] = {"ms_mean": ms, "ms_median": float(np.median(times)), "tokens_mean": float(np.mean(toks)),
                             "tokens_per_s": float(np.sum(toks) / (np.sum(times) / 1e3))}
    # the oracle: one layer over one 256-token sequence on the host
    import oracle as o
    p64 = [{k: v.double().cpu().numpy() for k, v in layers[0].items()}]
    x = np.random.default_rng(1).standard_normal((256, cfg.hidden))
    rel = shared["rel_embeddings"].double().cpu().numpy()
    t0 = time.perf_counter()
    o.encoder(x, p64, rel, np.ones(cfg.hidden), np.zeros(cfg.hidden), np.array([0, 256]), cfg.heads,
              buckets=cfg.buckets, max_rel=cfg.max_rel, span=cfg.span, eps=cfg.eps)
    cpu_tps = 256 / (time.perf_counter() - t0) / cfg.layers
    head = res["b1_l8192"]
    line = {"metric": "DeBERTa-v3-base encoder forward latency (12 layers, packed)", "value": head["ms_mean"],
            "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": False,
            "dtype": "bf16", "data": "synthetic (random weights; no checkpoint in the container)",
            "config": {"workload": "v3base_encoder_b1_l8192", "lengths": "uniform in [0.6 L, L]"},
            "workloads": res, "gpu_launches": None,
            "context": {"pages_h200_bf16_ms": {"b1_l8192": 39.35, "b16_l8192": 708.29},
                        "note": "the pages' figures: H200, trained weights; context, not a like-for-like target"},
            "cpu_baseline": {"value": cpu_tps, "unit": "tokens/s (12 layers)", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": "one layer over one 256-token sequence, float64 numpy"}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.op in ("pack", "linear", "encoder", "bwd", "small"):
        if rank == 0:
            {"pack": run_pack, "linear": run_linear, "encoder": run_encoder, "bwd": run_bwd,
             "small": run_small}[args.op](args, local)
        return
    assert args.warmup >= 3, "at least 3 warm-up steps"
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from exact_attention_deberta_gb300.build import build
    if rank == 0 or world == 1:
        build()
    if dist is not None:
        dist.barrier()
    from exact_attention_deberta_gb300 import binding, synth

    full = synth.make_inputs(args.workload)
    x = shard_inputs(full, rank, world)
    lengths = [int(n) for n in x.lengths]
    H, d, span = x.w.H, x.w.d, x.w.span
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=span)
    names = ("q", "k", "v", "pk", "pq", "key_mask", "cu_seqlens")
    host = {n: getattr(x, n) for n in names if getattr(x, n) is not None}
    dev = {n: t.cuda() for n, t in host.items()}
    out = torch.empty_like(dev["q"])
    B = len(x.lengths)
    fast32 = args.fp32_mode == "fast" and x.w.dtype == "fp32"
    size_fn = binding.df_attn_fwd_fp32_fast_workspace_size if fast32 else binding.df_attn_workspace_size
    fwd = binding.df_attn_fwd_fp32_fast if fast32 else binding.df_attn_fwd
    ws = torch.empty(size_fn(B, H, x.w.L, d, **kw), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step(inp, o):
        if x.w.layout == "packed":
            fwd(inp["q"], inp["k"], inp["v"], inp["pk"], inp["pq"], cu_seqlens=inp["cu_seqlens"],
                max_seqlen=x.w.L, out=o, workspace=ws, **kw)
        else:
            fwd(inp["q"], inp["k"], inp["v"], inp["pk"], inp["pq"], key_mask=inp["key_mask"], out=o,
                workspace=ws, **kw)

    for _ in range(args.warmup):
        step(dev, out)
    torch.cuda.synchronize()
    assert binding.df_attn_get_device_status(ws) == binding.DF_OK
    launches_per_step = binding.df_attn_last_launch_count()

    kev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
    for evs in kev:  # torch creates the CUDA events lazily, at their first record
        for e in evs:
            e.record(stream)
    # Inputs and output smaller than ~1.5x the 129 MB L2 would stay cached from
    # one step to the next: then every timed step is preceded by a 256 MB write
    # (outside its own events) and the steps are timed one by one.
    io_bytes = sum(t.numel() * t.element_size() for t in (dev["q"], dev["k"], dev["v"], out))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if io_bytes < 1.5 * L2_BYTES else None
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if flush is not None else 0)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(i & 255)
                sev[i][0].record(stream)
            binding.df_attn_set_profile_events(kev[i][0], kev[i][2])
            binding.df_attn_set_profile_split(kev[i][1])
            step(dev, out)
            if flush is not None:
                sev[i][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
    binding.df_attn_set_profile_events(None, None)
    binding.df_attn_set_profile_split(None)
    if dist is not None:
        dist.barrier()
    if flush is not None:
        ms = sum(a.elapsed_time(b) for a, b in sev) / args.steps
    else:
        ms = t0.elapsed_time(t1) / args.steps
    near_ms = sum(a.elapsed_time(m) for a, m, _ in kev) / args.steps
    far_ms = sum(m.elapsed_time(b) for _, m, b in kev) / args.steps
    hdr = ws[:64].view(torch.int32).cpu()
    rsp, rsn = int(hdr[3]), int(hdr[4])
    assert binding.df_attn_get_device_status(ws) == binding.DF_OK

    e2e = None
    numa = GpuLocalCpus(local)
    if not args.no_e2e and not fast32:
        numa.__enter__()
        # the host-buffer entry point: page-locked inputs and output (allocated
        # on the GPU's NUMA node), the copies of each group of sequences
        # overlapped with the kernels of another
        pinned = {n: t.pin_memory() for n, t in host.items()}
        out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in pinned.values())
        d2h = out_h.numel() * out_h.element_size()
        scratch = torch.empty(binding.df_attn_fwd_host_scratch_size(
            B, H, x.w.L, d, dev["q"].dtype, group_tokens=args.group_tokens, **kw), dtype=torch.uint8,
            device="cuda")

        def host_step():
            mode = (dict(cu_seqlens=pinned["cu_seqlens"], max_seqlen=x.w.L) if x.w.layout == "packed"
                    else dict(key_mask=pinned["key_mask"]))
            binding.df_attn_fwd_host(pinned["q"], pinned["k"], pinned["v"], pinned["pk"], pinned["pq"],
                                     out=out_h, group_tokens=args.group_tokens, scratch=scratch, **mode, **kw)

        for _ in range(2):
            host_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            host_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.steps
        assert binding.df_attn_get_device_status(scratch) == binding.DF_OK
        e2e = (e2e_ms, h2d, d2h)
        numa.__exit__(None, None, None)

    # max over ranks
    ms, near_ms, far_ms, e2e_ms = max_over_ranks([ms, near_ms, far_ms, e2e[0] if e2e else 0.0],
                                                 dist, device="cuda")

    # every rank processes one workload's worth on average: the job's units are
    # world x the workload's, whatever the split
    flops_rank = metric_flops(full.lengths, H, d)
    tokens_rank = float(sum(full.lengths))
    value = job_throughput(world, flops_rank, ms) / 1e12
    peaks, peak_src = load_peaks()
    # bf16 / fp16 run on the tensor cores (d = 32 as d = 64 on zero-widened heads;
    # the algorithmic count below keeps the true d)
    tc = x.w.dtype in ("bf16", "fp16") or fast32
    if tc:
        # the timed region is a fraction of a second at the maximum SM clock (the
        # clock record says so), not a seconds-long run under the power cap: the
        # burst dense rate applies; the sustained one is reported beside it (fp16
        # has the same dense rate as bf16)
        bound, peak, unit = "tensor", float(peaks["bf16_tflops"]), "TFLOP/s"
        near_algo, far_algo = tile_flops(lengths, H, d, span, rsp, rsn)
        near_file = "df_tc_near64.cu" if d in (32, 64) else "df_tc_near128.cu"
        if far_ms >= near_ms:
            kernel_file, kname, algo, kern_ms = "df_tc_far.cu", "tc_far_kernel", far_algo, far_ms
            other = ("tc_near_kernel", near_algo, near_ms)
        else:
            kernel_file, kname, algo, kern_ms = near_file, "tc_near_kernel", near_algo, near_ms
            other = ("tc_far_kernel", far_algo, far_ms)
    else:
        # FP32 FFMA: 152 SMs x 128 lanes x 2 flop x 2.07 GHz
        bound, peak, unit = "alu", 152 * 128 * 2 * 2.07e9 / 1e12, "TFLOP/s"
        kernel_file, kname = "df_simt.cu", "simt_fwd_kernel"
        algo, kern_ms, other = algorithmic_flops(lengths, H, d, span), far_ms, None
    achieved = algo / (kern_ms * 1e-3) / 1e12
    tr = traffic_record(kernel_file, x.w.name)
    line = {
        "metric": "disentangled-attn fwd TFLOP/s (8*L^2*d/head)",
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp16" if fast32 else (x.w.dtype if tc else "f32"),
        "data": "synthetic",
        "config": {"workload": x.w.name, "sequences": len(full.lengths), "seq_len": int(x.w.L),
                   "H": H, "d": d, "io_dtype": x.w.dtype, "layout": x.w.layout,
                   "fp32_mode": args.fp32_mode if x.w.dtype == "fp32" else None,
                   "buckets": x.w.buckets, "max_rel": x.w.max_rel, "span": span,
                   "sharding": ("one workload per rank" if world == 1 else
                                f"{world} workloads' sequences split over {world} ranks by n^2 cost"),
                   "l2": ("inputs larger than L2 (q,k,v,out %.0f MB)" % (io_bytes / 1e6)
                          if flush is None else
                          "L2 flushed before every timed step (256 MB write outside the step's "
                          "events; q,k,v,out %.0f MB)" % (io_bytes / 1e6))},
        "tokens_per_s": job_throughput(world, tokens_rank, ms),
        "pct_bf16_peak_metric": value / world / float(peaks["bf16_tflops"]) * 100.0,
        "pct_bf16_sustained_metric": value / world / float(peaks["bf16_tflops_sustained"]) * 100.0,
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": tr.get("dram_bytes_per_launch") if tr else None,
                     "kernel": kname, "kernel_ms": kern_ms, "algorithmic_flops": algo,
                     "peak_source": (peak_src + " bf16_tflops (burst)") if bound == "tensor" else
                     "derived: 152 SM x 128 FP32 lanes x 2 x 2.07 GHz"},
    }
    if bound == "tensor":
        sus = float(peaks["bf16_tflops_sustained"])
        line["roofline"]["peak_sustained"] = sus
        line["roofline"]["frac_sustained"] = achieved / sus
    if other is not None:
        oname, oalgo, oms = other
        line["roofline"]["other_kernel"] = {"kernel": oname, "kernel_ms": oms, "algorithmic_flops": oalgo,
                                            "achieved": oalgo / (oms * 1e-3) / 1e12,
                                            "frac": oalgo / (oms * 1e-3) / 1e12 / peak}
    if e2e:
        line["e2e"] = {"value": job_throughput(world, flops_rank, e2e_ms) / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": e2e[1], "d2h_bytes_per_step": e2e[2],
                       "host_numa_node": numa.node}
    clocks = clk.summary()
    line["clocks"] = clocks
    if rank == 0 and not args.no_cpu_baseline:
        tf, rows_s, rows, secs, thr = cpu_oracle_rate(x)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                                "sample": f"{rows} query rows of head 0 of one {int(lengths[0])}-token "
                                          f"sequence, float64 numpy, {secs:.1f} s"}
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
