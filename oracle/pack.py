"""Oracle of the padded <-> packed conversion.

TEST INFRASTRUCTURE ONLY (see the package header).  It follows DisentangledFlash
0.2.0 README, "Packed unpadded inference": right-padded [B, L, hidden] input
becomes FlashAttention-style [total_tokens, hidden] rows with cu_seqlens, and
the same metadata unpacks the output.  Reading taken where the README shows
only right padding: the valid positions of any 0/1 mask are taken in row-major
order, and unpacking writes zeros at the invalid positions.
"""

from __future__ import annotations

import numpy as np


def pack_info(mask: np.ndarray):
    """(cu_seqlens [B+1], indices [T], inverse [B*L], T, max_seqlen) of a mask [B, L]."""
    m = np.asarray(mask) != 0
    B, L = m.shape
    counts = m.sum(axis=1).astype(np.int64)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(counts)
    flat = m.reshape(-1)
    indices = np.flatnonzero(flat).astype(np.int32)          # row-major order
    inverse = np.full(B * L, -1, dtype=np.int32)
    inverse[indices] = np.arange(indices.size, dtype=np.int32)
    return cu, indices, inverse, int(indices.size), int(counts.max(initial=0))


def pack_rows(x: np.ndarray, indices: np.ndarray) -> np.ndarray:
    """tokens[k] = x[indices[k]] over the flattened padded rows."""
    rows = x.reshape(-1, x.shape[-1]) if x.ndim > 1 else x.reshape(-1, 1)
    return rows[np.asarray(indices, dtype=np.int64)]


def unpack_rows(tokens: np.ndarray, inverse: np.ndarray) -> np.ndarray:
    """out[r] = tokens[inverse[r]] where inverse[r] >= 0, else zeros; [B*L, row]."""
    inv = np.asarray(inverse, dtype=np.int64)
    out = np.zeros((inv.size,) + tokens.shape[1:], dtype=tokens.dtype)
    valid = inv >= 0
    out[valid] = tokens[inv[valid]]
    return out
