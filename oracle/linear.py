"""Oracle of the projections that feed the attention (float64).

TEST INFRASTRUCTURE ONLY (see the package header).  DisentangledFlash 0.2.0
README, "Status": the fused QKV projection (Q, K, V from one pass over the
hidden states) and the relative-position projections PK, PQ of the relative
embeddings; each output is x . W_i^T + b_i with W_i in the nn.Linear layout
[out_features, in_features].
"""

from __future__ import annotations

import numpy as np


def linear(x, weights, biases=None):
    """[x . W_i^T + b_i for each W_i] in float64 (x [M, K], W_i [N, K], b_i [N] or None)."""
    x64 = np.asarray(x, dtype=np.float64)
    outs = []
    for i, w in enumerate(weights):
        y = x64 @ np.asarray(w, dtype=np.float64).T
        if biases is not None and biases[i] is not None:
            y = y + np.asarray(biases[i], dtype=np.float64)[None, :]
        outs.append(y)
    return outs
