"""Plain float64 oracle for exact DeBERTa-v2/v3 disentangled attention (forward).

TEST INFRASTRUCTURE ONLY -- imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference arm, never by the product path.
It shares no code, table or constant with the CUDA library.

What is computed (sources):

* DisentangledFlash 0.2.0 README, section "Status": bidirectional
  DeBERTa-v2/v3 attention with C2P/P2C disentangled terms, factorized 2-D
  padding masks, packed inference with ``cu_seqlens``; the attention matrix
  is never materialised by the fast path (the oracle does materialise it,
  one head and one row chunk at a time).
* kernels-community discussion "DisentangledFlash", section "Motivation":
  the score adds a content-to-position and a position-to-content term to
  the content-to-content dot product, and the fast kernel evaluates the
  same formulation exactly (no approximation).

Neither page writes the formula out.  The readings used here (each is
listed with its reason in the design notes):

  score(i, j) = ( Q_i . K_j  +  Q_i . PK[idx(i-j)]  +  K_j . PQ[idx(i-j)] ) / sqrt(3 d)
  idx(r)      = clamp(bucket(r) + span, 0, 2 span - 1)
  bucket(r)   = r                                   if |r| <= mid  (mid = buckets // 2)
              = sign(r) (mid + ceil(ln(|r|/mid) / ln((max_rel-1)/mid) (mid-1)))   otherwise
  bucket(r)   = r  for every r when buckets <= 0

* the p2c term uses the same index as the c2p term (bucket is odd, so the
  "negate, gather, transpose" form of the position-to-content term lands on
  idx(i-j));
* the factorized mask m (1 = valid) removes key j when m_j = 0 and sets the
  whole output row i to zero when m_i = 0;
* positions are token indices inside a sequence (padded: 0..L-1 of the batch
  row; packed: restart at 0 at every cu_seqlens boundary).

Parity pins for every function live in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import math

import numpy as np

# Largest [rows, n] float64 block the oracle materialises at once.
_BLOCK_BYTES = 256 << 20


def log_bucket(r, buckets: int, max_rel: int) -> np.ndarray:
    """DeBERTa log-bucketed relative position, evaluated in float64.

    Identity inside |r| <= buckets // 2; logarithmic growth outside it, so
    that |r| = max_rel - 1 lands exactly on bucket 2 * mid - 1.  With
    ``buckets <= 0`` the relative position is used as is.
    """
    r = np.asarray(r, dtype=np.int64)
    out = r.copy()
    if buckets <= 0:
        return out
    mid = buckets // 2
    a = np.abs(r)
    far = a > mid
    if np.any(far):
        af = a[far].astype(np.float64)
        frac = np.log(af / mid) / np.log((max_rel - 1) / mid)
        grown = np.ceil(frac * (mid - 1)).astype(np.int64) + mid
        out[far] = np.sign(r[far]) * grown
    return out


def rel_index(r, buckets: int, max_rel: int, span: int) -> np.ndarray:
    """Row of PK / PQ used for relative distance r = i - j."""
    return np.clip(log_bucket(r, buckets, max_rel) + span, 0, 2 * span - 1)


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (any dtype) -> float64 numpy
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def attend_rows(q, k, v, pk, pq, head: int, rows, *, buckets, max_rel, span,
                valid=None) -> np.ndarray:
    """Output rows ``rows`` of one head of one sequence.

    q, k, v: [n, H, d]; pk, pq: [2 span, H, d]; valid: optional bool [n]
    (the factorized mask).  Returns [len(rows), d] float64.
    """
    q = _as_f64(q)[:, head]
    k = _as_f64(k)[:, head]
    v = _as_f64(v)[:, head]
    pk = _as_f64(pk)[:, head]
    pq = _as_f64(pq)[:, head]
    n, d = q.shape
    rows = np.asarray(rows, dtype=np.int64)
    if valid is None:
        valid = np.ones(n, dtype=bool)
    valid = np.asarray(valid, dtype=bool)
    scale = 1.0 / math.sqrt(3.0 * d)
    out = np.zeros((rows.size, d), dtype=np.float64)
    if rows.size == 0 or n == 0:
        return out
    c2p = q[rows] @ pk.T                 # [m, 2 span]  content -> position
    p2c = k @ pq.T                       # [n, 2 span]  position -> content
    keys = np.arange(n)
    chunk = max(1, _BLOCK_BYTES // (8 * max(n, 1)))
    for c0 in range(0, rows.size, chunk):
        rr = rows[c0:c0 + chunk]
        idx = rel_index(rr[:, None] - keys[None, :], buckets, max_rel, span)
        z = q[rr] @ k.T
        z += np.take_along_axis(c2p[c0:c0 + chunk], idx, axis=1)
        z += p2c[keys[None, :], idx]
        z *= scale
        z[:, ~valid] = -np.inf
        live = valid[rr]
        if not np.any(live):
            continue
        zl = z[live]
        zl -= zl.max(axis=1, keepdims=True)
        p = np.exp(zl)
        p /= p.sum(axis=1, keepdims=True)
        blk = np.zeros((rr.size, d), dtype=np.float64)
        blk[live] = p @ v
        out[c0:c0 + chunk] = blk
    return out


def attend_sequence(q, k, v, pk, pq, *, buckets, max_rel, span, valid=None):
    """All heads, all rows of one sequence: [n, H, d] -> [n, H, d] float64."""
    q = _as_f64(q)
    n, H, d = q.shape
    out = np.zeros((n, H, d), dtype=np.float64)
    rows = np.arange(n)
    for h in range(H):
        out[:, h] = attend_rows(q, k, v, pk, pq, h, rows, buckets=buckets,
                                max_rel=max_rel, span=span, valid=valid)
    return out


def attend_padded(q, k, v, pk, pq, key_mask, *, buckets, max_rel, span):
    """Padded layout: q, k, v [B, L, H, d]; key_mask [B, L] (nonzero = valid)."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    mask = np.asarray(key_mask.cpu().numpy() if hasattr(key_mask, "cpu") else key_mask) != 0
    B = q.shape[0]
    out = np.zeros_like(q)
    for b in range(B):
        out[b] = attend_sequence(q[b], k[b], v[b], pk, pq, buckets=buckets,
                                 max_rel=max_rel, span=span, valid=mask[b])
    return out


def attend_packed(q, k, v, pk, pq, cu_seqlens, *, buckets, max_rel, span):
    """Packed layout: q, k, v [T, H, d]; cu_seqlens [S + 1] int."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    cu = np.asarray(cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                    dtype=np.int64)
    out = np.zeros_like(q)
    for s in range(cu.size - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        out[a:b] = attend_sequence(q[a:b], k[a:b], v[a:b], pk, pq, buckets=buckets,
                                   max_rel=max_rel, span=span)
    return out


def metric_flops(lengths, H: int, d: int) -> float:
    """Throughput metric's work count: 8 n^2 d per head over valid tokens."""
    return float(sum(8.0 * float(n) * float(n) * d * H for n in lengths))
