"""Oracle of a DeBERTa-v3 encoder on the packed layout (float64).

TEST INFRASTRUCTURE ONLY (see the package header).  The pages' benchmark
workload is the 12-layer DeBERTa-v3-base encoder (DisentangledFlash README,
"Benchmarks": encoder latency with projections and FFN included).  A layer,
as the README's packed path runs it: the fused QKV projection; PK and PQ from
the key and query projections of the layer-normalised relative embeddings
(shared attention keys); disentangled attention; the output projection with a
residual LayerNorm; a GELU feed-forward block with a residual LayerNorm.
"""

from __future__ import annotations

import numpy as np
from scipy.special import erf

from .df_oracle import attend_packed
from .linear import linear


def layer_norm(x, gamma, beta, eps):
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def gelu(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def encoder_layer(h, p, rel, cu_seqlens, heads, *, buckets, max_rel, span, eps):
    """One layer on packed rows h [T, hidden]; p holds the layer's weights as
    float64 arrays (w_qkv [3 hidden, hidden], b_qkv, w_o, b_o, ln1_g, ln1_b,
    w_1 [4 hidden, hidden], b_1, w_2 [hidden, 4 hidden], b_2, ln2_g, ln2_b)."""
    T, hid = h.shape
    d = hid // heads
    w, b = p["w_qkv"], p["b_qkv"]
    q, k, v = linear(h, [w[:hid], w[hid:2 * hid], w[2 * hid:]], [b[:hid], b[hid:2 * hid], b[2 * hid:]])
    pk, pq = linear(rel, [w[hid:2 * hid], w[:hid]], [b[hid:2 * hid], b[:hid]])
    ctx = attend_packed(q.reshape(T, heads, d), k.reshape(T, heads, d), v.reshape(T, heads, d),
                        pk.reshape(-1, heads, d), pq.reshape(-1, heads, d), cu_seqlens,
                        buckets=buckets, max_rel=max_rel, span=span)
    (a,) = linear(ctx.reshape(T, hid), [p["w_o"]], [p["b_o"]])
    h1 = layer_norm(a + h, p["ln1_g"], p["ln1_b"], eps)
    (f,) = linear(h1, [p["w_1"]], [p["b_1"]])
    (f2,) = linear(gelu(f), [p["w_2"]], [p["b_2"]])
    return layer_norm(f2 + h1, p["ln2_g"], p["ln2_b"], eps)


def encoder(h, layers, rel_embeddings, rel_g, rel_b, cu_seqlens, heads, *, buckets, max_rel, span, eps):
    rel = layer_norm(rel_embeddings, rel_g, rel_b, eps)
    out = np.asarray(h, dtype=np.float64)
    for p in layers:
        out = encoder_layer(out, p, rel, cu_seqlens, heads, buckets=buckets, max_rel=max_rel, span=span,
                            eps=eps)
    return out
