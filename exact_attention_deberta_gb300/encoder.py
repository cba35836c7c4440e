"""A DeBERTa-v3 encoder on the packed layout, composed from the library's
calls (every step runs in libdfattn.so; this module only orders the calls and
holds the weights).

The pages' benchmark workload is the 12-layer DeBERTa-v3-base encoder
(DisentangledFlash README, "Benchmarks").  A layer: the fused QKV projection
(df_linear, three outputs in the attention's [T, H, d] layout); PK and PQ from
the layer's key and query projections of the layer-normalised relative
embeddings (shared attention keys); disentangled attention (df_attn_fwd,
packed); the output projection and a residual LayerNorm; the feed-forward
block (projection with GELU, projection) and a residual LayerNorm.
Weights are synthetic (no checkpoint is available): N(0, 0.02) matrices,
N(0, 0.02) biases, LayerNorm gain 1 and shift 0.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List

import torch

from . import binding


@dataclass
class EncoderConfig:
    hidden: int = 768
    heads: int = 12
    layers: int = 12
    ffn: int = 3072
    buckets: int = 256
    max_rel: int = 512
    eps: float = 1e-7

    @property
    def span(self):
        return binding.default_span(self.buckets, self.max_rel)


def synthetic_weights(cfg: EncoderConfig, dtype=torch.bfloat16, device="cuda", seed=0):
    g = torch.Generator().manual_seed(seed)

    def rnd(*shape, std=0.02):
        return (torch.randn(*shape, generator=g) * std).to(dtype).to(device)

    def ones(n):
        return torch.ones(n, dtype=dtype, device=device)

    def zeros(n):
        return torch.zeros(n, dtype=dtype, device=device)

    h, f = cfg.hidden, cfg.ffn
    layers = [dict(w_qkv=rnd(3 * h, h), b_qkv=rnd(3 * h), w_o=rnd(h, h), b_o=rnd(h), ln1_g=ones(h), ln1_b=zeros(h),
                   w_1=rnd(f, h), b_1=rnd(f), w_2=rnd(h, f), b_2=rnd(h), ln2_g=ones(h), ln2_b=zeros(h))
              for _ in range(cfg.layers)]
    shared = dict(rel_embeddings=rnd(2 * cfg.span, h), rel_g=ones(h), rel_b=zeros(h))
    return layers, shared


class Encoder:
    """encoder(hidden [T, hidden], cu_seqlens [S + 1], max_seqlen) -> [T, hidden]."""

    def __init__(self, cfg: EncoderConfig, layers: List[dict], shared: dict):
        self.cfg, self.layers, self.shared = cfg, layers, shared

    def __call__(self, hidden, cu_seqlens, max_seqlen, stream=None, trace=None):
        """``trace``: an optional list; each layer appends a dict of the tensors
        its attention call took and gave (q, k, v, pk, pq, ctx), which the layer
        computes anyway (nothing extra runs)."""
        cfg = self.cfg
        hid, H = cfg.hidden, cfg.heads
        T = hidden.shape[0]
        sh = self.shared
        rel = binding.df_layernorm(sh["rel_embeddings"], sh["rel_g"], sh["rel_b"], eps=cfg.eps, stream=stream)
        ws = None
        h = hidden
        for p in self.layers:
            w, b = p["w_qkv"], p["b_qkv"]
            q, k, v = binding.qkv_projection(h, w, b, H, stream=stream)
            pk, pq = binding.rel_projection(rel, w[hid:2 * hid], b[hid:2 * hid], w[:hid], b[:hid], H, stream=stream)
            if ws is None:
                size = binding.df_attn_workspace_size(cu_seqlens.numel() - 1, H, max_seqlen, hid // H,
                                                      cfg.buckets, cfg.max_rel, cfg.span)
                ws = torch.empty(max(size, 256), dtype=torch.uint8, device=hidden.device)
            ctx = binding.df_attn_fwd(q, k, v, pk, pq, cu_seqlens=cu_seqlens, max_seqlen=max_seqlen,
                                      buckets=cfg.buckets, max_rel=cfg.max_rel, span=cfg.span, workspace=ws,
                                      stream=stream)
            if trace is not None:
                trace.append(dict(q=q, k=k, v=v, pk=pk, pq=pq, ctx=ctx))
            (a,) = binding.df_linear(ctx.view(T, hid), [p["w_o"]], [p["b_o"]], stream=stream)
            h1 = binding.df_layernorm(a, p["ln1_g"], p["ln1_b"], residual=h, eps=cfg.eps, stream=stream)
            (f,) = binding.df_linear(h1, [p["w_1"]], [p["b_1"]], stream=stream, activation=binding.LINEAR_GELU)
            (f2,) = binding.df_linear(f, [p["w_2"]], [p["b_2"]], stream=stream)
            h = binding.df_layernorm(f2, p["ln2_g"], p["ln2_b"], residual=h1, eps=cfg.eps, stream=stream)
        return h
