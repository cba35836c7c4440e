"""Pins of the encoder oracle's parts (oracle/encoder.py) against closed forms:
LayerNorm gives zero mean and unit variance rows and a hand-computed case;
GELU at 0, +-1 (x times the standard normal CDF) and far out; a layer whose
weights and biases are all zero reduces to LayerNorm of its input (no
attention contribution, GELU(0) = 0)."""

import math

import numpy as np

from oracle import encoder_layer, gelu, layer_norm


def test_layer_norm_rows_are_standardised():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((6, 256)) * 3 + 1
    y = layer_norm(x, np.ones(256), np.zeros(256), 0.0)
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=1), 1, atol=1e-10)


def test_layer_norm_hand_case():
    y = layer_norm(np.array([[1.0, 2.0, 3.0]]), np.array([2.0, 2.0, 2.0]), np.array([0.0, 1.0, 0.0]), 1e-7)
    s = math.sqrt(2.0 / 3.0 + 1e-7)
    np.testing.assert_allclose(y, [[-2.0 / s, 1.0, 2.0 / s]], rtol=1e-12)


def test_gelu_values():
    phi1 = 0.5 * (1 + math.erf(1 / math.sqrt(2)))
    np.testing.assert_allclose(gelu(np.array([0.0, 1.0, -1.0, 30.0, -30.0])),
                               [0.0, phi1, -(1 - phi1), 30.0, 0.0], rtol=1e-12, atol=1e-12)


def test_zero_weight_layer_is_layer_norm_of_input():
    hid, H, T = 256, 4, 40
    rng = np.random.default_rng(1)
    h = rng.standard_normal((T, hid))
    z = np.zeros
    p = dict(w_qkv=z((3 * hid, hid)), b_qkv=z(3 * hid), w_o=z((hid, hid)), b_o=z(hid), ln1_g=np.ones(hid),
             ln1_b=z(hid), w_1=z((4 * hid, hid)), b_1=z(4 * hid), w_2=z((hid, 4 * hid)), b_2=z(hid),
             ln2_g=np.ones(hid), ln2_b=z(hid))
    rel = rng.standard_normal((512, hid))
    out = encoder_layer(h, p, rel, np.array([0, 25, 40]), H, buckets=256, max_rel=512, span=256, eps=1e-7)
    np.testing.assert_allclose(out, layer_norm(h, np.ones(hid), z(hid), 1e-7), atol=1e-6)


def test_one_wrong_head_fails_the_per_head_attention_bound():
    """The GPU encoder test checks every head's attention output per layer
    (relative L2 <= 1e-2, the bf16 attention tolerance) besides the final
    hidden states (mean |err| < 1e-2, max < 0.15).  With the encoder's synthetic
    weights a mistake confined to one head of twelve moves the final states by
    about 2e-3 on average and 2e-2 at most, inside that bound; planted in the
    oracle, each plausible mistake (a position term dropped, PK and PQ swapped,
    the content term lost) moves that head's attention output by more than ten
    times the per-head bound."""
    import torch
    from oracle import attend_packed, linear
    from exact_attention_deberta_gb300.encoder import EncoderConfig, synthetic_weights
    cfg = EncoderConfig(hidden=768, heads=12, layers=2, ffn=3072)
    layers, shared = synthetic_weights(cfg, device="cpu", seed=5)
    lengths = [300, 150, 77]
    T, hid, H = sum(lengths), cfg.hidden, cfg.heads
    d = hid // H
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    g = torch.Generator().manual_seed(9)
    h = torch.randn(T, hid, generator=g).to(torch.bfloat16).double().numpy()
    p = {k: v.double().numpy() for k, v in layers[0].items()}
    rel = layer_norm(shared["rel_embeddings"].double().numpy(), shared["rel_g"].double().numpy(),
                     shared["rel_b"].double().numpy(), cfg.eps)
    w, b = p["w_qkv"], p["b_qkv"]
    q, k, v = linear(h, [w[:hid], w[hid:2 * hid], w[2 * hid:]], [b[:hid], b[hid:2 * hid], b[2 * hid:]])
    pk, pq = linear(rel, [w[hid:2 * hid], w[:hid]], [b[hid:2 * hid], b[:hid]])
    q, k, v = (t.reshape(T, H, d) for t in (q, k, v))
    pk, pq = pk.reshape(-1, H, d), pq.reshape(-1, H, d)
    kw = dict(buckets=cfg.buckets, max_rel=cfg.max_rel, span=cfg.span)
    right = attend_packed(q, k, v, pk, pq, cu, **kw)
    planted = {"no c2p": (q, k, v, 0 * pk, pq), "no p2c": (q, k, v, pk, 0 * pq),
               "PK and PQ swapped": (q, k, v, pq, pk), "no content term": (q, 0 * k, v, pk, pq)}
    for name, args in planted.items():
        wrong = attend_packed(*args, cu, **kw)
        rel_err = np.linalg.norm(wrong[:, 5] - right[:, 5]) / np.linalg.norm(right[:, 5])
        assert rel_err > 10 * 1e-2, (name, rel_err)
