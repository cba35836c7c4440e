"""Plain float64 oracle for the backward pass of disentangled attention.

TEST INFRASTRUCTURE ONLY -- used by ``tests/`` and ``bench.py``'s CPU arm,
never by the product path; it shares no code with the CUDA library.

The pages have no backward pass (DisentangledFlash 0.2.0 README, "Status":
training still takes the stock DeBERTa path).  This module differentiates
the forward that ``df_oracle`` evaluates, by the chain rule written out step
by step for one head of one sequence:

  z_ij   = scale * (Q_i.K_j + Q_i.PK[idx_ij] + K_j.PQ[idx_ij]),  scale = 1/sqrt(3 d)
  p_ij   = softmax over valid keys j of z_ij;  O_i = sum_j p_ij V_j   (valid rows)

  dV_j   = sum_i p_ij dO_i
  dP_ij  = dO_i . V_j
  dz_ij  = p_ij (dP_ij - sum_k p_ik dP_ik)
  dS_ij  = scale * dz_ij                      (gradient of the raw score)
  dQ_i   = sum_j dS_ij (K_j + PK[idx_ij])
  dK_j   = sum_i dS_ij (Q_i + PQ[idx_ij])
  dPK[r] = sum_{i,j: idx_ij = r} dS_ij Q_i
  dPQ[r] = sum_{i,j: idx_ij = r} dS_ij K_j

An output row whose query is masked is the constant 0, so it passes no
gradient; a masked key has p = 0 in every row.  The position sums go
through the bucket-summed matrices G_c2p[i, r] = sum_{j: idx_ij = r} dS_ij
and G_p2c[j, r] = sum_{i: idx_ij = r} dS_ij (a library bincount), so that
dQ gets G_c2p . PK and dPK = G_c2p^T . Q, and likewise on the key side.

Pins: ``tests/test_backward_oracle.py`` (central differences of the forward
oracle, shift invariances of the score, the reduction to the library's
scaled-dot-product attention when PK = PQ = 0, masked rows and keys).
"""

from __future__ import annotations

import math

import numpy as np

from .df_oracle import _as_f64, rel_index

_BLOCK_BYTES = 256 << 20


def backward_head(q, k, v, pk, pq, dout, *, buckets, max_rel, span, valid=None):
    """Gradients of one head of one sequence.

    q, k, v, dout: [n, d]; pk, pq: [2 span, d]; valid: optional bool [n].
    Returns (dq, dk, dv, dpk, dpq) as float64 arrays of the inputs' shapes.
    """
    q, k, v, pk, pq, dout = (_as_f64(a) for a in (q, k, v, pk, pq, dout))
    n, d = q.shape
    R = 2 * span
    dq = np.zeros((n, d))
    dk = np.zeros((n, d))
    dv = np.zeros((n, d))
    dpk = np.zeros((R, d))
    dpq = np.zeros((R, d))
    if n == 0:
        return dq, dk, dv, dpk, dpq
    valid = np.ones(n, dtype=bool) if valid is None else np.asarray(valid, dtype=bool)
    scale = 1.0 / math.sqrt(3.0 * d)
    c2p = q @ pk.T                      # [n, 2 span]
    p2c = k @ pq.T                      # [n, 2 span]
    keys = np.arange(n)
    g_c2p = np.zeros((n, R))
    g_p2c = np.zeros((n, R))
    chunk = max(1, _BLOCK_BYTES // (8 * n))
    for c0 in range(0, n, chunk):
        rr = np.arange(c0, min(n, c0 + chunk))
        live = valid[rr]
        if not np.any(live):
            continue
        rr = rr[live]
        m = rr.size
        idx = rel_index(rr[:, None] - keys[None, :], buckets, max_rel, span)
        z = q[rr] @ k.T + np.take_along_axis(c2p[rr], idx, axis=1) + p2c[keys[None, :], idx]
        z *= scale
        z[:, ~valid] = -np.inf
        z -= z.max(axis=1, keepdims=True)
        p = np.exp(z)
        p /= p.sum(axis=1, keepdims=True)
        dP = dout[rr] @ v.T
        dz = p * (dP - (p * dP).sum(axis=1, keepdims=True))
        dS = scale * dz                 # zero at masked keys, since p is
        dv += p.T @ dout[rr]
        dq[rr] += dS @ k
        dk += dS.T @ q[rr]
        # bucket sums along the relative index
        rows = np.repeat(np.arange(m), n)
        flat = idx.ravel()
        g_c2p[rr] += np.bincount(rows * R + flat, weights=dS.ravel(), minlength=m * R).reshape(m, R)
        cols = np.tile(keys, m)
        g_p2c += np.bincount(cols * R + flat, weights=dS.ravel(), minlength=n * R).reshape(n, R)
    dq += g_c2p @ pk
    dk += g_p2c @ pq
    dpk += g_c2p.T @ q
    dpq += g_p2c.T @ k
    return dq, dk, dv, dpk, dpq


def _row_softmax(q, k, v, pk, pq, rr, keys, valid, scale, buckets, max_rel, span):
    """Scores, softmax and output of query rows rr (all keys of the head)."""
    idx = rel_index(rr[:, None] - keys[None, :], buckets, max_rel, span)
    z = q[rr] @ k.T + np.einsum("md,mnd->mn", q[rr], pk[idx]) + np.einsum("nd,mnd->mn", k, pq[idx])
    z *= scale
    z[:, ~valid] = -np.inf
    z -= z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    return idx, p, p @ v


def backward_rows(q, k, v, pk, pq, dout, rows, *, buckets, max_rel, span, valid=None):
    """dQ of the given query rows of one head: [n, d] inputs -> [len(rows), d].

    A row's dQ needs only its own softmax row: dS_ij = scale p_ij (dO_i.V_j -
    dO_i.O_i) and dQ_i = sum_j dS_ij (K_j + PK[idx_ij]).
    """
    q, k, v, pk, pq, dout = (_as_f64(a) for a in (q, k, v, pk, pq, dout))
    n, d = q.shape
    valid = np.ones(n, dtype=bool) if valid is None else np.asarray(valid, dtype=bool)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, d))
    live = valid[rows]
    if not np.any(live):
        return out
    rr = rows[live]
    scale = 1.0 / math.sqrt(3.0 * d)
    keys = np.arange(n)
    idx, p, o = _row_softmax(q, k, v, pk, pq, rr, keys, valid, scale, buckets, max_rel, span)
    dS = scale * p * (dout[rr] @ v.T - np.sum(dout[rr] * o, axis=1, keepdims=True))
    out[live] = dS @ k + np.einsum("mn,mnd->md", dS, pk[idx])
    return out


def backward_keys(q, k, v, pk, pq, dout, keys_sel, *, buckets, max_rel, span, valid=None):
    """(dK, dV) of the given keys of one head: [n, d] inputs -> two [m, d].

    Every valid query row's softmax is needed (its normaliser and D_i), one
    row chunk at a time; only the selected key columns are kept.
    """
    q, k, v, pk, pq, dout = (_as_f64(a) for a in (q, k, v, pk, pq, dout))
    n, d = q.shape
    valid = np.ones(n, dtype=bool) if valid is None else np.asarray(valid, dtype=bool)
    sel = np.asarray(keys_sel, dtype=np.int64)
    dk = np.zeros((sel.size, d))
    dv = np.zeros((sel.size, d))
    scale = 1.0 / math.sqrt(3.0 * d)
    keys = np.arange(n)
    rows_all = np.nonzero(valid)[0]
    c2p = q @ pk.T
    p2c = k @ pq.T
    chunk = max(1, _BLOCK_BYTES // (8 * max(n, 1)))
    for c0 in range(0, rows_all.size, chunk):
        rr = rows_all[c0:c0 + chunk]
        idx = rel_index(rr[:, None] - keys[None, :], buckets, max_rel, span)
        z = q[rr] @ k.T + np.take_along_axis(c2p[rr], idx, axis=1) + p2c[keys[None, :], idx]
        z *= scale
        z[:, ~valid] = -np.inf
        z -= z.max(axis=1, keepdims=True)
        p = np.exp(z)
        p /= p.sum(axis=1, keepdims=True)
        o = p @ v
        dmean = np.sum(dout[rr] * o, axis=1, keepdims=True)
        ps = p[:, sel]
        dS = scale * ps * (dout[rr] @ v[sel].T - dmean)
        dv += ps.T @ dout[rr]
        dk += dS.T @ q[rr] + np.einsum("ms,msd->sd", dS, pq[idx[:, sel]])
    dk[~valid[sel]] = 0.0
    dv[~valid[sel]] = 0.0
    return dk, dv


def backward_sequence(q, k, v, pk, pq, dout, *, buckets, max_rel, span, valid=None):
    """All heads of one sequence: [n, H, d] inputs, [2 span, H, d] positions."""
    q, k, v, pk, pq, dout = (_as_f64(a) for a in (q, k, v, pk, pq, dout))
    n, H, d = q.shape
    grads = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v),
             np.zeros_like(pk), np.zeros_like(pq)]
    for h in range(H):
        parts = backward_head(q[:, h], k[:, h], v[:, h], pk[:, h], pq[:, h], dout[:, h],
                              buckets=buckets, max_rel=max_rel, span=span, valid=valid)
        for g, part in zip(grads, parts):
            g[:, h] = part
    return tuple(grads)


def backward_padded(q, k, v, pk, pq, dout, key_mask, *, buckets, max_rel, span):
    """Padded layout [B, L, H, d]; the position gradients sum over the batch."""
    q, k, v, dout = (_as_f64(a) for a in (q, k, v, dout))
    mask = np.asarray(key_mask.cpu().numpy() if hasattr(key_mask, "cpu") else key_mask) != 0
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dpk = np.zeros(np.shape(pk))
    dpq = np.zeros(np.shape(pq))
    for b in range(q.shape[0]):
        g = backward_sequence(q[b], k[b], v[b], pk, pq, dout[b], buckets=buckets,
                              max_rel=max_rel, span=span, valid=mask[b])
        dq[b], dk[b], dv[b] = g[0], g[1], g[2]
        dpk += g[3]
        dpq += g[4]
    return dq, dk, dv, dpk, dpq


def backward_packed(q, k, v, pk, pq, dout, cu_seqlens, *, buckets, max_rel, span):
    """Packed layout [T, H, d] with cu_seqlens [S + 1]."""
    q, k, v, dout = (_as_f64(a) for a in (q, k, v, dout))
    cu = np.asarray(cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                    dtype=np.int64)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dpk = np.zeros(np.shape(pk))
    dpq = np.zeros(np.shape(pq))
    for s in range(cu.size - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        g = backward_sequence(q[a:b], k[a:b], v[a:b], pk, pq, dout[a:b], buckets=buckets,
                              max_rel=max_rel, span=span)
        dq[a:b], dk[a:b], dv[a:b] = g[0], g[1], g[2]
        dpk += g[3]
        dpq += g[4]
    return dq, dk, dv, dpk, dpq


def backward_metric_flops(lengths, H: int, d: int) -> float:
    """Work count of the backward: 22 n^2 d per head.

    Eleven n x n x d products of the direct formulation: the three score
    terms recomputed, dP, dV, dQ, dK, and the four position sums (into dQ,
    dK, dPK and dPQ), two flops each.
    """
    return float(sum(22.0 * float(n) * float(n) * d * H for n in lengths))
