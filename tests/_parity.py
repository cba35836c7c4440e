"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the float64 oracle on the same rounded inputs, compare."""

from __future__ import annotations

import numpy as np
import torch

from oracle import attend_padded, attend_packed, attend_rows

# Tolerances (max-abs, rel-L2) per I/O dtype.
TOL = {"bf16": (3e-2, 1e-2), "fp16": (1e-2, 3e-3), "fp32": (1e-5, 1e-5)}


def to_dev(x):
    return None if x is None else x.cuda()


def run_gpu(binding, x, *, out=None, workspace=None, dev_inputs=None):
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    d = dev_inputs or {n: to_dev(getattr(x, n)) for n in ("q", "k", "v", "pk", "pq", "key_mask",
                                                          "cu_seqlens")}
    check_status = workspace is None
    if workspace is None:
        B = d["q"].shape[0] if x.w.layout == "padded" else d["cu_seqlens"].numel() - 1
        size = binding.df_attn_workspace_size(B, x.w.H, x.w.L, x.w.d, **kw)
        workspace = torch.empty(max(size, 256), dtype=torch.uint8, device="cuda")
    if x.w.layout == "padded":
        o = binding.df_attn_fwd(d["q"], d["k"], d["v"], d["pk"], d["pq"], key_mask=d["key_mask"],
                                out=out, workspace=workspace, **kw)
    else:
        o = binding.df_attn_fwd(d["q"], d["k"], d["v"], d["pk"], d["pq"],
                                cu_seqlens=d["cu_seqlens"], max_seqlen=x.w.L, out=out,
                                workspace=workspace, **kw)
    torch.cuda.synchronize()
    if check_status:
        st = binding.df_attn_get_device_status(workspace)
        assert st == binding.DF_OK, f"device status {binding.status_string(st)}"
    return o


def oracle_full(x) -> np.ndarray:
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    if x.w.layout == "padded":
        return attend_padded(x.q, x.k, x.v, x.pk, x.pq, x.key_mask, **kw)
    return attend_packed(x.q, x.k, x.v, x.pk, x.pq, x.cu_seqlens, **kw)


def sample_triples(x, count: int, seed: int):
    """Seeded (sequence, head, row) triples over valid query rows."""
    rng = np.random.default_rng(seed)
    seqs = [(s, st, n) for s, (st, n) in enumerate(x.seq_slices()) if n > 0]
    out = []
    for _ in range(count):
        s, st, n = seqs[int(rng.integers(len(seqs)))]
        out.append((s, int(rng.integers(x.w.H)), int(rng.integers(n))))
    # always include the first / last rows of the longest sequence (tile edges)
    s, st, n = max(seqs, key=lambda t: t[2])
    out += [(s, 0, 0), (s, x.w.H - 1, n - 1), (s, 0, min(n - 1, 127)), (s, 0, min(n - 1, 128))]
    return out


def oracle_sampled(x, triples):
    """Oracle rows for the sampled triples: dict (token, head) -> [d] float64."""
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    slices = x.seq_slices()
    groups = {}
    for s, h, r in triples:
        groups.setdefault((s, h), set()).add(r)
    res = {}
    for (s, h), rows in groups.items():
        st, n = slices[s]
        rows = np.array(sorted(rows))
        if x.w.layout == "padded":
            b = s
            valid = x.key_mask[b, :n].numpy() != 0
            sl = lambda t: t[b, :n]  # noqa: E731
        else:
            valid = None
            sl = lambda t: t[st:st + n]  # noqa: E731
        o = attend_rows(sl(x.q), sl(x.k), sl(x.v), x.pk, x.pq, h, rows, valid=valid, **kw)
        for r, val in zip(rows, o):
            res[(st + int(r), h)] = val
    return res


def gpu_rows(x, out, keys):
    flat = out.reshape(-1, x.w.H, x.w.d)
    idx_t = torch.tensor([k[0] for k in keys], device=out.device)
    idx_h = torch.tensor([k[1] for k in keys], device=out.device)
    return flat[idx_t, idx_h].double().cpu().numpy()


def errors(got: np.ndarray, ref: np.ndarray):
    diff = np.abs(got - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    return max_abs, rel


def assert_close(got, ref, dtype: str, what: str = ""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    max_abs, rel = errors(got, ref)
    tmax, trel = TOL[dtype]
    assert max_abs <= tmax and rel <= trel, (
        f"{what}: max-abs {max_abs:.3e} (tol {tmax:g}), rel-L2 {rel:.3e} (tol {trel:g})")
    return max_abs, rel
