"""Pins of the float64 oracle against facts that do not come from the oracle.

Each test ties one part of the oracle to something fixed independently of it:
hand-derived closed forms (tests/golden/log_bucket_anchors.txt), analytic
attention patterns whose softmax can be written down by hand, a library
routine (torch's scaled-dot-product attention in float64) for the case the
method reduces to, and invariants of the formula.  A dropped term, a wrong
sign of the relative distance, a wrong index offset or a swapped projection
each fails at least one of them.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import attend_packed, attend_padded, attend_rows, attend_sequence, log_bucket, rel_index

HERE = os.path.dirname(os.path.abspath(__file__))


def _anchors():
    rows = []
    with open(os.path.join(HERE, "golden", "log_bucket_anchors.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            p = line.split()
            rows.append(tuple(int(x) for x in (p[0], p[1], p[2], p[3], p[5], p[6])))
    return rows


@pytest.mark.parametrize("buckets,max_rel,span,r,bucket,idx", _anchors())
def test_bucket_anchor(buckets, max_rel, span, r, bucket, idx):
    assert int(log_bucket(np.array([r]), buckets, max_rel)[0]) == bucket
    assert int(rel_index(np.array([r]), buckets, max_rel, span)[0]) == idx


@pytest.mark.parametrize("buckets,max_rel", [(256, 512), (64, 128), (8, 16), (32, 4096)])
def test_bucket_identity_zone_and_shape(buckets, max_rel):
    mid = buckets // 2
    r = np.arange(-mid, mid + 1)
    assert np.array_equal(log_bucket(r, buckets, max_rel), r)
    r = np.arange(-9000, 9001)
    b = log_bucket(r, buckets, max_rel)
    assert np.array_equal(b[::-1], -b)                 # odd
    assert np.all(np.diff(b) >= 0)                     # non-decreasing
    # closed form: |r| = max_rel - 1 lands on 2 mid - 1 exactly
    assert int(log_bucket(np.array([max_rel - 1]), buckets, max_rel)[0]) == 2 * mid - 1
    # strictly inside the log zone the bucket moves slower than r
    far = r[(r > mid)]
    assert np.all(log_bucket(far, buckets, max_rel) <= far)


def test_no_buckets_is_identity():
    r = np.arange(-3000, 3001)
    assert np.array_equal(log_bucket(r, 0, 512), r)
    assert np.array_equal(log_bucket(r, -1, 512), r)


def test_index_saturation_points_deberta_defaults():
    r = np.arange(-8191, 8192)
    idx = rel_index(r, 256, 512, 256)
    assert idx.min() == 0 and idx.max() == 511
    assert np.unique(idx).size == 512
    assert r[idx == 511].min() == 506          # hand-derived: 505 -> 510, 506 -> 511
    assert r[idx == 0].max() == -512           # hand-derived: -511 -> 1, -512 -> 0


def test_bucket_precision_is_moot_for_defaults():
    """fp32 evaluation (as a float32 host would do it) gives the same buckets."""
    mid, max_rel = 128, 512
    a = np.arange(mid + 1, 8192, dtype=np.int64)
    f32 = np.ceil(np.log(a.astype(np.float32) / np.float32(mid))
                  / np.log(np.float32((max_rel - 1) / mid)) * np.float32(mid - 1)) + mid
    assert np.array_equal(f32.astype(np.int64), log_bucket(a, 256, max_rel))


def _one_hot_case(n, d, *, a, kind):
    """Inputs whose logits are  a  at j = i - 1 (kind 'c2p' or 'p2c') and 0 elsewhere."""
    span = 256
    rng = np.random.default_rng(123)
    s = math.sqrt(3.0 * d)
    v = rng.standard_normal((n, 1, d))
    pk = rng.standard_normal((2 * span, 1, d))
    pq = rng.standard_normal((2 * span, 1, d))
    e0 = np.zeros(d)
    e0[0] = 1.0
    if kind == "c2p":
        q = np.tile(e0, (n, 1))[:, None, :]
        k = np.zeros((n, 1, d))
        pk[:] = 0.0
        pk[span + 1, 0] = a * s * e0           # r = i - j = +1  ->  idx = span + 1
    else:
        q = np.zeros((n, 1, d))
        k = np.tile(e0, (n, 1))[:, None, :]
        pq[:] = 0.0
        pq[span + 1, 0] = a * s * e0
    return q, k, v, pk, pq


@pytest.mark.parametrize("kind", ["c2p", "p2c"])
def test_relative_direction_closed_form(kind):
    n, d, a = 6, 4, 2.5
    q, k, v, pk, pq = _one_hot_case(n, d, a=a, kind=kind)
    out = attend_sequence(q, k, v, pk, pq, buckets=256, max_rel=512, span=256)[:, 0]
    V = v[:, 0]
    exp_a = math.exp(a)
    for i in range(n):
        if i == 0:  # no key at distance +1: all logits equal
            want = V.mean(axis=0)
        else:
            want = (exp_a * V[i - 1] + V.sum(axis=0) - V[i - 1]) / (exp_a + n - 1)
        np.testing.assert_allclose(out[i], want, rtol=0, atol=1e-13)


def test_terms_add_closed_form():
    """Q.K constant, c2p at r=+1 and p2c at r=-1: both biases appear, summed."""
    n, d, span = 7, 4, 256
    s = math.sqrt(3.0 * d)
    rng = np.random.default_rng(7)
    e0 = np.zeros(d)
    e0[0] = 1.0
    q = np.tile(e0, (n, 1))[:, None, :]
    k = np.tile(e0, (n, 1))[:, None, :]
    v = rng.standard_normal((n, 1, d))
    pk = np.zeros((2 * span, 1, d))
    pq = np.zeros((2 * span, 1, d))
    a, b = 1.7, -0.9
    pk[span + 1, 0] = a * s * e0
    pq[span - 1, 0] = b * s * e0
    out = attend_sequence(q, k, v, pk, pq, buckets=256, max_rel=512, span=span)[:, 0]
    V = v[:, 0]
    for i in range(n):
        w = np.ones(n)
        if i - 1 >= 0:
            w[i - 1] = math.exp(a)
        if i + 1 < n:
            w[i + 1] = math.exp(b)
        np.testing.assert_allclose(out[i], w @ V / w.sum(), rtol=0, atol=1e-13)


@pytest.mark.parametrize("masked", [False, True])
def test_zero_positions_reduce_to_sdpa(masked):
    """PK = PQ = 0: plain softmax attention at scale 1/sqrt(3 d) (torch, float64)."""
    rng = np.random.default_rng(11)
    B, L, H, d = 2, 40, 3, 16
    q = rng.standard_normal((B, L, H, d))
    k = rng.standard_normal((B, L, H, d))
    v = rng.standard_normal((B, L, H, d))
    pk = np.zeros((512, H, d))
    pq = np.zeros((512, H, d))
    mask = np.ones((B, L), dtype=np.uint8)
    if masked:
        mask[0, 29:] = 0
        mask[1, 3] = 0
        mask[1, 17:25] = 0
    out = attend_padded(q, k, v, pk, pq, mask, buckets=256, max_rel=512, span=256)
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    keep = torch.from_numpy(mask != 0)
    attn_mask = keep[:, None, None, :].expand(B, H, L, L)
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=attn_mask, scale=1.0 / math.sqrt(3 * d)).permute(0, 2, 1, 3).numpy()
    live = mask != 0
    np.testing.assert_allclose(out[live], ref[live], rtol=0, atol=1e-12)
    assert np.all(out[~live] == 0.0)


def _rand_seq(n, H, d, span=256, seed=5):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s)  # noqa: E731
    return f(n, H, d), f(n, H, d), f(n, H, d), f(2 * span, H, d), f(2 * span, H, d)


def test_equal_pk_rows_do_not_matter():
    q, k, v, pk, pq = _rand_seq(50, 2, 8)
    pk_a = np.broadcast_to(pk[:1], pk.shape).copy()
    pk_b = np.zeros_like(pk)
    kw = dict(buckets=256, max_rel=512, span=256)
    np.testing.assert_allclose(attend_sequence(q, k, v, pk_a, pq, **kw),
                               attend_sequence(q, k, v, pk_b, pq, **kw), rtol=0, atol=1e-12)
    # ...whereas equal PQ rows still matter (the p2c bias varies with the key)
    pq_a = np.broadcast_to(pq[:1], pq.shape).copy()
    assert not np.allclose(attend_sequence(q, k, v, pk, pq_a, **kw),
                           attend_sequence(q, k, v, pk, np.zeros_like(pq), **kw))


def test_constant_values_and_single_token():
    q, k, v, pk, pq = _rand_seq(33, 2, 8)
    c = np.random.default_rng(1).standard_normal((1, 2, 8))
    vc = np.broadcast_to(c, v.shape).copy()
    out = attend_sequence(q, k, vc, pk, pq, buckets=256, max_rel=512, span=256)
    np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), rtol=0, atol=1e-13)
    out1 = attend_sequence(q[:1], k[:1], v[:1], pk, pq, buckets=256, max_rel=512, span=256)
    np.testing.assert_allclose(out1, v[:1], rtol=0, atol=1e-15)


def test_masked_tokens_do_not_leak():
    rng = np.random.default_rng(3)
    B, L, H, d = 2, 64, 2, 8
    q, k, v = (rng.standard_normal((B, L, H, d)) for _ in range(3))
    pk, pq = (rng.standard_normal((512, H, d)) for _ in range(2))
    mask = np.ones((B, L), dtype=np.uint8)
    mask[0, 41:] = 0
    mask[1, 5:9] = 0
    kw = dict(buckets=256, max_rel=512, span=256)
    ref = attend_padded(q, k, v, pk, pq, mask, **kw)
    dead = mask == 0
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for x in (q2, k2, v2):
        x[dead] = 1e3 * rng.standard_normal(x[dead].shape)
    got = attend_padded(q2, k2, v2, pk, pq, mask, **kw)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    assert np.all(got[dead] == 0.0)


def test_packed_equals_padded():
    rng = np.random.default_rng(9)
    lens = [5, 64, 1, 37]
    H, d, L = 2, 8, 64
    kw = dict(buckets=256, max_rel=512, span=256)
    pk, pq = (rng.standard_normal((512, H, d)) for _ in range(2))
    T = sum(lens)
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    cu = np.concatenate([[0], np.cumsum(lens)])
    packed = attend_packed(q, k, v, pk, pq, cu, **kw)
    pad = lambda x: np.stack([np.pad(x[cu[s]:cu[s + 1]], ((0, L - lens[s]), (0, 0), (0, 0)))  # noqa
                              for s in range(len(lens))])
    mask = np.zeros((len(lens), L), dtype=np.uint8)
    for s, n in enumerate(lens):
        mask[s, :n] = 1
    padded = attend_padded(pad(q), pad(k), pad(v), pk, pq, mask, **kw)
    for s, n in enumerate(lens):
        np.testing.assert_allclose(packed[cu[s]:cu[s + 1]], padded[s, :n], rtol=0, atol=1e-12)


def test_unreachable_position_rows_do_not_matter():
    """n = 128 with (256, 512, 256): only idx in [129, 383] can be reached."""
    q, k, v, pk, pq = _rand_seq(128, 1, 8)
    kw = dict(buckets=256, max_rel=512, span=256)
    r = np.arange(-127, 128)
    reach = np.unique(rel_index(r, 256, 512, 256))
    assert reach.min() == 129 and reach.max() == 383
    ref = attend_sequence(q, k, v, pk, pq, **kw)
    other = np.setdiff1d(np.arange(512), reach)
    pk2, pq2 = pk.copy(), pq.copy()
    pk2[other] = 50.0
    pq2[other] = -50.0
    np.testing.assert_allclose(attend_sequence(q, k, v, pk2, pq2, **kw), ref, rtol=0, atol=1e-13)


def _brute(q, k, v, pk, pq, valid, buckets, max_rel, span):
    """Scalar triple loop with the bucket taken from the hand-anchored function."""
    n, H, d = q.shape
    out = np.zeros((n, H, d))
    s = 1.0 / math.sqrt(3 * d)
    for h in range(H):
        for i in range(n):
            if not valid[i]:
                continue
            logits = []
            for j in range(n):
                if not valid[j]:
                    logits.append(-math.inf)
                    continue
                u = int(rel_index(np.array([i - j]), buckets, max_rel, span)[0])
                acc = 0.0
                for t in range(d):
                    acc += q[i, h, t] * k[j, h, t] + q[i, h, t] * pk[u, h, t] + k[j, h, t] * pq[u, h, t]
                logits.append(acc * s)
            m = max(logits)
            w = [math.exp(x - m) if x != -math.inf else 0.0 for x in logits]
            z = sum(w)
            for j in range(n):
                out[i, h] += w[j] / z * v[j, h]
    return out


@pytest.mark.parametrize("buckets,max_rel,span,n", [(8, 16, 8, 23), (256, 512, 256, 17), (0, 6, 6, 15)])
def test_vectorised_gathers_match_scalar_loop(buckets, max_rel, span, n):
    rng = np.random.default_rng(n)
    H, d = 2, 3
    q, k, v = (rng.standard_normal((n, H, d)) for _ in range(3))
    pk, pq = (rng.standard_normal((2 * span, H, d)) for _ in range(2))
    valid = np.ones(n, dtype=bool)
    valid[[2, 7]] = False
    got = attend_sequence(q, k, v, pk, pq, buckets=buckets, max_rel=max_rel, span=span, valid=valid)
    want = _brute(q, k, v, pk, pq, valid, buckets, max_rel, span)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    rows = np.array([0, 3, n - 1])
    part = attend_rows(q, k, v, pk, pq, 1, rows, buckets=buckets, max_rel=max_rel, span=span,
                       valid=valid)
    np.testing.assert_allclose(part, want[rows, 1], rtol=0, atol=1e-12)
