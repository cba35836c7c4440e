"""Backward pass through the C ABI against the float64 backward oracle.

Small cases (several 64-row tiles, ragged tails, masked holes, empty and
one-token sequences, near and far tiles, every dtype and head size) are
compared element by element on every gradient.  At the long packed workload
(16 x 8192 tokens, H = 12, d = 64, and H = 8, d = 128) the oracle computes
sampled rows of dQ and sampled keys of dK and dV one by one, and the position
gradients are checked
through identities that hold at any size:
  sum_r dPK[r] = 0                      (a shift of every PK row moves no softmax)
  sum_j dV_j = sum_i dO_i               (softmax rows sum to one)
  sum dK.K - sum dPQ.PQ = sum dQ.Q - sum dPK.PK   (both are sum_ij dS_ij Q_i.K_j)
all per head.

Tolerance: every gradient is computed in fp32 from the same rounded inputs
the oracle reads, so the gap is fp32 rounding of sums over up to a few
thousand terms: max |gpu - oracle| <= 2e-4 * max |oracle| per tensor.
"""

import numpy as np
import pytest
import torch

from exact_attention_deberta_gb300 import synth
from oracle import backward_keys, backward_packed, backward_padded, backward_rows

pytestmark = pytest.mark.gpu

TOL = 2e-4


def _kw(x):
    return dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)


def _run(lib, x, dout):
    d = [getattr(x, n).cuda() for n in ("q", "k", "v", "pk", "pq")]
    g = dout.cuda()
    if x.w.layout == "padded":
        res = lib.df_attn_bwd(*d, g, key_mask=x.key_mask.cuda(), **_kw(x))
    else:
        res = lib.df_attn_bwd(*d, g, cu_seqlens=x.cu_seqlens.cuda(), max_seqlen=x.w.L, **_kw(x))
    torch.cuda.synchronize()
    return [r.cpu().double().numpy() for r in res]


def _oracle(x, dout):
    if x.w.layout == "padded":
        return backward_padded(x.q, x.k, x.v, x.pk, x.pq, dout, x.key_mask, **_kw(x))
    return backward_packed(x.q, x.k, x.v, x.pk, x.pq, dout, x.cu_seqlens, **_kw(x))


def _close(name, got, ref, tol=TOL):
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    scale = max(float(np.abs(ref).max()), 1e-30)
    err = float(np.abs(got - ref).max()) / scale
    assert err <= tol, f"{name}: max error {err:.2e} of max |ref| {scale:.3e}"


CASES = {
    # right padding, near and far tiles (saturation at |r| >= 63), strict fp32
    "padded_fp32_d64_far": dict(layout="padded", dtype="fp32", H=2, d=64, lengths=[97, 300], L=300,
                                buckets=16, max_rel=64),
    # one-token and tile-edge lengths, default DeBERTa-v3 buckets (all tiles near)
    "packed_bf16_d64_edges": dict(layout="packed", dtype="bf16", H=3, d=64, lengths=[1, 64, 129, 300],
                                  buckets=256, max_rel=512),
    "packed_bf16_d128_far": dict(layout="packed", dtype="bf16", H=2, d=128, lengths=[200, 77],
                                 buckets=16, max_rel=64),
    # an empty sequence among others, head size 32
    "packed_fp16_d32_empty": dict(layout="packed", dtype="fp16", H=2, d=32, lengths=[150, 0, 65],
                                  buckets=32, max_rel=128),
    # no bucketing: span = max_rel = 128
    "padded_bf16_nobuckets": dict(layout="padded", dtype="bf16", H=2, d=64, lengths=[130, 64], L=192,
                                  buckets=0, max_rel=128),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_matches_oracle(lib, name):
    x = synth.custom_inputs(seed=5, **CASES[name])
    if x.w.layout == "padded":
        x.key_mask[0, [5, 40, 41]] = 0   # holes inside the sequence, not only right padding
    dout = synth.grad_output(x)
    got = _run(lib, x, dout)
    ref = _oracle(x, dout)
    for nm, g, r in zip(("dq", "dk", "dv", "dpk", "dpq"), got, ref):
        _close(f"{name}/{nm}", g, r)
    if x.w.layout == "padded":
        dead = x.key_mask.numpy() == 0
        for nm, g in zip(("dq", "dk", "dv"), got[:3]):
            assert np.all(g[dead] == 0.0), f"{nm}: masked tokens must get exact zeros"


def test_backward_without_buckets_span_512(lib):
    """DeBERTa without position buckets: span = max_rel = 512 (1024 PK / PQ rows)."""
    x = synth.custom_inputs(layout="packed", dtype="bf16", H=2, d=64, lengths=[700, 90], buckets=0,
                            max_rel=512, seed=8)
    dout = synth.grad_output(x)
    got = _run(lib, x, dout)
    ref = _oracle(x, dout)
    for nm, g, r in zip(("dq", "dk", "dv", "dpk", "dpq"), got, ref):
        _close(f"nobuckets512/{nm}", g, r)


def _identities(x, dout, got, tol=TOL):
    dq, dk, dv, dpk, dpq = got
    q, k, pk, pq, g = (t.double().numpy() for t in (x.q, x.k, x.pk, x.pq, dout))
    for h in range(x.w.H):
        scale = np.abs(dpk[:, h]).sum(axis=0).max() + 1e-30
        assert np.abs(dpk[:, h].sum(axis=0)).max() <= tol * scale, f"sum dPK head {h}"
        sv = g[:, h].sum(axis=0)
        assert np.abs(dv[:, h].sum(axis=0) - sv).max() <= tol * (np.abs(g[:, h]).sum(axis=0).max()), h
        terms = [np.sum(dk[:, h] * k[:, h]), np.sum(dpq[:, h] * pq[:, h]),
                 np.sum(dq[:, h] * q[:, h]), np.sum(dpk[:, h] * pk[:, h])]
        mag = (np.abs(dk[:, h] * k[:, h]).sum() + np.abs(dpq[:, h] * pq[:, h]).sum()
               + np.abs(dq[:, h] * q[:, h]).sum() + np.abs(dpk[:, h] * pk[:, h]).sum())
        gap = (terms[0] - terms[1]) - (terms[2] - terms[3])
        assert abs(gap) <= tol * mag, f"gradient identity head {h}: gap {gap:.3e} of {mag:.3e}"


@pytest.mark.slow
@pytest.mark.parametrize("workload", ["long_packed_h12d64", "long_packed_h8d128"])
def test_backward_long_packed_sampled(lib, workload):
    x = synth.make_inputs(workload)
    dout = synth.grad_output(x)
    got = _run(lib, x, dout)
    for nm, g in zip(("dq", "dk", "dv", "dpk", "dpq"), got):
        assert np.all(np.isfinite(g)), nm
    _identities(x, dout, got)
    rng = np.random.default_rng(21)
    slices = x.seq_slices()
    for s, h in [(0, 0), (int(rng.integers(len(slices))), int(rng.integers(x.w.H)))]:
        st, n = slices[s]
        sl = slice(st, st + n)
        args = [t[sl, h] for t in (x.q, x.k, x.v)] + [x.pk[:, h], x.pq[:, h], dout[sl, h]]
        rows = np.unique(np.concatenate([[0, 63, 64, 127, 128, n - 1], rng.integers(0, n, 4)]))
        ref = backward_rows(*args, rows, **_kw(x))
        _close(f"dq rows seq {s} head {h}", got[0][st + rows, h], ref)
        keys = np.unique(np.concatenate([[0, 64, n - 1], rng.integers(0, n, 2)]))
        rk, rv = backward_keys(*args, keys, **_kw(x))
        _close(f"dk keys seq {s} head {h}", got[1][st + keys, h], rk)
        _close(f"dv keys seq {s} head {h}", got[2][st + keys, h], rv)
