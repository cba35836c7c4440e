"""Pins of the float64 backward oracle against facts that do not come from it.

* Central differences of the forward oracle (itself pinned in
  test_oracle_pins.py): every entry of every gradient on a small head whose
  distances reach the identity zone, the log zone and saturation, and
  directional derivatives on padded (masked) and packed batches.
* Shift invariances of the score: adding one vector to every PK row adds
  Q_i.u to the whole row i of scores, so the softmax (and the loss) does not
  move and sum_r dPK[r] = 0; with PQ = 0 the same holds for K.  Also
  sum_j dV_j = sum_i dO_i over valid rows, since each softmax row sums to 1.
* With PK = PQ = 0 the method is plain attention with scale 1/sqrt(3 d):
  dQ, dK, dV equal torch's scaled-dot-product attention gradients (float64
  autograd, a library routine).
* Masked query rows and masked keys get zero gradients.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attend_packed, attend_padded, attend_sequence
from oracle.backward import (backward_head, backward_keys, backward_packed, backward_padded,
                             backward_rows, backward_sequence)

CFG = dict(buckets=4, max_rel=8, span=4)   # mid 2: identity |r| <= 2, log zone, saturation at 7


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _loss_seq(q, k, v, pk, pq, w, valid=None):
    return float(np.sum(attend_sequence(q, k, v, pk, pq, valid=valid, **CFG) * w))


def test_every_entry_matches_central_differences():
    rng = np.random.default_rng(11)
    n, H, d = 10, 1, 3
    q, k, v, w = (_rand(rng, n, H, d) for _ in range(4))
    pk, pq = (_rand(rng, 2 * CFG["span"], H, d) for _ in range(2))
    valid = np.ones(n, dtype=bool)
    valid[[3, 8]] = False   # one masked row/key inside, one near the end
    grads = backward_sequence(q, k, v, pk, pq, w, valid=valid, **CFG)
    args = [q, k, v, pk, pq]
    eps = 1e-6
    for which, (x, g) in enumerate(zip(args, grads)):
        num = np.zeros_like(x)
        for e in np.ndindex(x.shape):
            old = x[e]
            x[e] = old + eps
            up = _loss_seq(*args, w, valid)
            x[e] = old - eps
            dn = _loss_seq(*args, w, valid)
            x[e] = old
            num[e] = (up - dn) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8, err_msg=f"input {which}")


def _directional(loss, args, grads, rng, eps=1e-6):
    for which, (x, g) in enumerate(zip(args, grads)):
        u = rng.standard_normal(x.shape)
        x0 = x.copy()
        x[...] = x0 + eps * u
        up = loss()
        x[...] = x0 - eps * u
        dn = loss()
        x[...] = x0
        fd = (up - dn) / (2 * eps)
        an = float(np.sum(g * u))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (which, fd, an)


def test_padded_directional_derivatives():
    rng = np.random.default_rng(12)
    B, L, H, d = 2, 12, 2, 4
    q, k, v, w = (_rand(rng, B, L, H, d) for _ in range(4))
    pk, pq = (_rand(rng, 2 * CFG["span"], H, d) for _ in range(2))
    mask = np.ones((B, L), dtype=np.uint8)
    mask[0, 9:] = 0          # right padding
    mask[1, [0, 5]] = 0      # holes
    grads = backward_padded(q, k, v, pk, pq, w, mask, **CFG)
    args = [q, k, v, pk, pq]

    def loss():
        return float(np.sum(attend_padded(*args, mask, **CFG) * w))

    _directional(loss, args, grads, rng)
    # masked tokens: no gradient into their q, k, v
    for g in grads[:3]:
        assert np.all(g[mask == 0] == 0.0)


def test_packed_directional_derivatives():
    rng = np.random.default_rng(13)
    cu = np.array([0, 5, 6, 17])   # lengths 5, 1, 11
    T, H, d = 17, 2, 4
    q, k, v, w = (_rand(rng, T, H, d) for _ in range(4))
    pk, pq = (_rand(rng, 2 * CFG["span"], H, d) for _ in range(2))
    grads = backward_packed(q, k, v, pk, pq, w, cu, **CFG)
    args = [q, k, v, pk, pq]

    def loss():
        return float(np.sum(attend_packed(*args, cu, **CFG) * w))

    _directional(loss, args, grads, rng)


def test_position_shift_invariance():
    rng = np.random.default_rng(14)
    n, d = 40, 8
    cfg = dict(buckets=16, max_rel=32, span=16)
    q, k, v, w = (_rand(rng, n, d) for _ in range(4))
    pk, pq = (_rand(rng, 32, d) for _ in range(2))
    valid = rng.random(n) > 0.2
    dq, dk, dv, dpk, dpq = backward_head(q, k, v, pk, pq, w, valid=valid, **cfg)
    np.testing.assert_allclose(dpk.sum(axis=0), 0.0, atol=1e-10)
    np.testing.assert_allclose(dv.sum(axis=0), w[valid].sum(axis=0), rtol=1e-10, atol=1e-10)
    # with PQ = 0 the key side has the same invariance
    dq, dk, dv, dpk, dpq = backward_head(q, k, v, pk, np.zeros_like(pq), w, valid=valid, **cfg)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-10)
    assert np.abs(dpq).max() > 0   # PQ = 0 still has a gradient


def test_reduces_to_library_attention_without_positions():
    rng = np.random.default_rng(15)
    n, d = 33, 16
    q, k, v, w = (_rand(rng, n, d) for _ in range(4))
    zeros = np.zeros((2 * 64, d))
    dq, dk, dv, _, _ = backward_head(q, k, v, zeros, zeros, w, buckets=64, max_rel=128, span=64)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], scale=1.0 / math.sqrt(3 * d))[0, 0]
    out.backward(torch.tensor(w, dtype=torch.float64))
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("n", [0, 1])
def test_degenerate_lengths(n):
    rng = np.random.default_rng(16)
    d = 4
    q, k, v, w = (_rand(rng, n, d) for _ in range(4))
    pk, pq = (_rand(rng, 8, d) for _ in range(2))
    dq, dk, dv, dpk, dpq = backward_head(q, k, v, pk, pq, w, **CFG)
    # one token attends only to itself with weight 1: O = V, every score gradient is 0
    assert np.all(dq == 0) and np.all(dk == 0) and np.all(dpk == 0) and np.all(dpq == 0)
    np.testing.assert_array_equal(dv, w)


def test_row_and_key_helpers_match_the_full_backward():
    rng = np.random.default_rng(17)
    n, d = 70, 8
    cfg = dict(buckets=16, max_rel=32, span=16)
    q, k, v, w = (_rand(rng, n, d) for _ in range(4))
    pk, pq = (_rand(rng, 32, d) for _ in range(2))
    valid = rng.random(n) > 0.15
    dq, dk, dv, _, _ = backward_head(q, k, v, pk, pq, w, valid=valid, **cfg)
    rows = np.array([0, 5, 33, 69, int(np.nonzero(~valid)[0][0])])
    np.testing.assert_allclose(backward_rows(q, k, v, pk, pq, w, rows, valid=valid, **cfg), dq[rows],
                               rtol=1e-10, atol=1e-12)
    bk, bv = backward_keys(q, k, v, pk, pq, w, rows, valid=valid, **cfg)
    np.testing.assert_allclose(bk, dk[rows], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(bv, dv[rows], rtol=1e-10, atol=1e-12)


def test_gradient_product_identity():
    """sum dK.K - sum dPQ.PQ = sum dQ.Q - sum dPK.PK (both are sum_ij dS_ij Q_i.K_j)."""
    rng = np.random.default_rng(18)
    n, d = 50, 6
    cfg = dict(buckets=16, max_rel=32, span=16)
    q, k, v, w = (_rand(rng, n, d) for _ in range(4))
    pk, pq = (_rand(rng, 32, d) for _ in range(2))
    dq, dk, dv, dpk, dpq = backward_head(q, k, v, pk, pq, w, **cfg)
    lhs = np.sum(dk * k) - np.sum(dpq * pq)
    rhs = np.sum(dq * q) - np.sum(dpk * pk)
    assert abs(lhs - rhs) < 1e-10 * (1 + abs(lhs))


def test_packed_and_padded_layouts_agree():
    """The same sequences as padded batch rows and as a packed batch give the
    same per-token gradients and the same position gradients."""
    rng = np.random.default_rng(19)
    lengths = [7, 12, 3]
    L, H, d = 12, 2, 4
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T = int(cu[-1])
    q, k, v, w = (_rand(rng, T, H, d) for _ in range(4))
    pk, pq = (_rand(rng, 2 * CFG["span"], H, d) for _ in range(2))
    packed = backward_packed(q, k, v, pk, pq, w, cu, **CFG)
    pad = lambda x: np.stack([np.concatenate([x[cu[b]:cu[b + 1]], np.zeros((L - n, H, d))])  # noqa: E731
                              for b, n in enumerate(lengths)])
    mask = np.zeros((len(lengths), L), dtype=np.uint8)
    for b, n in enumerate(lengths):
        mask[b, :n] = 1
    padded = backward_padded(pad(q), pad(k), pad(v), pk, pq, pad(w), mask, **CFG)
    for b, n in enumerate(lengths):
        for g_pk, g_pd in zip(packed[:3], padded[:3]):
            np.testing.assert_allclose(g_pd[b, :n], g_pk[cu[b]:cu[b + 1]], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(padded[3], packed[3], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(padded[4], packed[4], rtol=1e-12, atol=1e-12)


# Parity bound for a backward whose contractions run on the tensor cores with
# P and dS rounded to bf16 as MMA operands (fp32 accumulation; the bucket sums
# of dS, and with them dPK and dPQ, stay in fp32): written down before such a
# kernel exists.  Each rounded operand carries a relative error of at most the
# bf16 unit roundoff 2^-9; the bound is four times that, relative to the
# largest entry of the oracle's gradient.
TC_BWD_TOL = {"dq": 4 * 2.0 ** -9, "dk": 4 * 2.0 ** -9, "dv": 4 * 2.0 ** -9, "dpk": 2e-4, "dpq": 2e-4}


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _backward_bf16_operands(q, k, v, pk, pq, dout, *, buckets, max_rel, span, rounded_o=False):
    """The gradients of one head as such a kernel forms them: the exact
    softmax and dS (the chain rule of the module docstring), then P and dS
    rounded to bf16 wherever they enter a contraction (dV = P^T dO,
    dQ = dS K, dK = dS^T Q), the bucket sums of dS unrounded.  With
    rounded_o, D_i = dO_i . O_i takes the forward's output rounded to bf16."""
    from oracle import rel_index
    n, d = q.shape
    R, scale = 2 * span, 1.0 / math.sqrt(3.0 * d)
    keys = np.arange(n)
    idx = rel_index(keys[:, None] - keys[None, :], buckets, max_rel, span)
    z = q @ k.T + np.take_along_axis(q @ pk.T, idx, axis=1) + (k @ pq.T)[keys[None, :], idx]
    z = scale * z
    z -= z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    dP = dout @ v.T
    if rounded_o:
        dS = scale * p * (dP - (dout * _bf16(p @ v)).sum(axis=1, keepdims=True))
    else:
        dS = scale * p * (dP - (p * dP).sum(axis=1, keepdims=True))
    pb, dSb = _bf16(p), _bf16(dS)
    g_c2p = np.zeros((n, R))
    g_p2c = np.zeros((n, R))
    np.add.at(g_c2p, (np.repeat(keys, n), idx.ravel()), dS.ravel())
    np.add.at(g_p2c, (np.tile(keys, n), idx.ravel()), dS.ravel())
    return (dSb @ k + g_c2p @ pk, dSb.T @ q + g_p2c @ pq, pb.T @ dout, g_c2p.T @ q, g_p2c.T @ k)


@pytest.mark.parametrize("n,d,sigma,seed", [(300, 64, 1.0, 1), (500, 64, 4.0, 5), (400, 128, 2.0, 6)])
def test_bf16_operand_backward_stays_within_its_bound(n, d, sigma, seed):
    """bf16 inputs with distances through the identity zone, the log zone and
    saturation (DeBERTa's 256 / 512 / 256); the bf16-operand gradients stay
    within TC_BWD_TOL of the oracle, and dQ, dK, dV would not meet the fp32
    kernels' 2e-4 bound (so the looser one is needed, not just allowed)."""
    rng = np.random.default_rng(seed)
    q, k, pk, pq = (_bf16(rng.standard_normal(s) * sigma) for s in ((n, d), (n, d), (512, d), (512, d)))
    v, dout = (_bf16(rng.standard_normal((n, d))) for _ in range(2))
    kw = dict(buckets=256, max_rel=512, span=256)
    exact = backward_head(q, k, v, pk, pq, dout, **kw)
    rounded = _backward_bf16_operands(q, k, v, pk, pq, dout, **kw)
    worst_main = 0.0
    for name, a, b in zip(("dq", "dk", "dv", "dpk", "dpq"), exact, rounded):
        rel = np.abs(a - b).max() / np.abs(a).max()
        assert rel <= TC_BWD_TOL[name], (name, rel)
        if name in ("dq", "dk", "dv"):
            worst_main = max(worst_main, rel)
    assert worst_main > 2e-4


def test_d_from_the_rounded_output_breaks_the_position_gradients():
    """D_i = dO_i . O_i must come from an fp32 O: taken from the bf16-rounded
    forward output, its error enters every dS of the row and the position
    gradients (bucket sums of dS) leave their 2e-4 bound -- already for N(0, 1)
    inputs, and by more than ten times with sigma = 4."""
    kw = dict(buckets=256, max_rel=512, span=256)
    for n, sigma, seed, factor in ((400, 1.0, 7, 1.0), (500, 4.0, 5, 10.0)):
        rng = np.random.default_rng(seed)
        q, k, pk, pq = (_bf16(rng.standard_normal(s) * sigma) for s in ((n, 64), (n, 64), (512, 64), (512, 64)))
        v, dout = (_bf16(rng.standard_normal((n, 64))) for _ in range(2))
        exact = backward_head(q, k, v, pk, pq, dout, **kw)
        rounded = _backward_bf16_operands(q, k, v, pk, pq, dout, rounded_o=True, **kw)
        worst_pos = max(np.abs(a - b).max() / np.abs(a).max() for a, b in zip(exact[3:], rounded[3:]))
        assert worst_pos > factor * TC_BWD_TOL["dpk"], (sigma, worst_pos)
