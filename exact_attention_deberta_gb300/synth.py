"""Seeded synthetic inputs shaped like the DisentangledFlash workloads.

This module draws random numbers and casts them to the I/O dtype; it holds
none of the attention arithmetic.  Both the CUDA path and the float64 oracle
consume exactly the tensors produced here (the oracle upcasts the *rounded*
values).

Recipe (per workload): ``numpy.random.default_rng(seed)``; draw the sequence
lengths first, then Q, K, V, PK, PQ as float32 N(0, 1) in that order, then
cast to the workload dtype with round-to-nearest-even.  Layouts are
contiguous: padded ``[B, L, H, d]`` with a right-padded ``uint8 [B, L]``
key mask, packed ``[T, H, d]`` with ``int32 cu_seqlens [S + 1]``, and the
relative-position projections ``[2 span, H, d]``.

The workloads stand in for the DisentangledFlash README's DeBERTa-v3-base
encoder benchmark (section "Benchmark configuration": packed lengths,
B = 1 / 16, L up to 8192) and its MNLI run (section "Pretrained-model
parity": DeBERTa-v2-xlarge, B = 16, L = 512, 92.62 % padding).  Neither the
dataset nor the trained checkpoints are used: only their shapes.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    layout: str           # "padded" | "packed"
    dtype: str            # "bf16" | "fp16" | "fp32"
    H: int
    d: int
    L: int                # padded length, or the longest packed sequence bound
    batch: int            # batch rows (padded) or number of sequences (packed)
    lengths: str          # length law, see draw_lengths()
    buckets: int = 256
    max_rel: int = 512
    span: int = 256


WORKLOADS = {
    # tiny fp32 case, full length and with a key-padding length of 97
    "tiny_fp32": Workload("tiny_fp32", 0, "padded", "fp32", 2, 64, 128, 1, "full"),
    "tiny_fp32_pad97": Workload("tiny_fp32_pad97", 0, "padded", "fp32", 2, 64, 128, 1, "first97"),
    # DeBERTa-v3-base-shaped padded batch
    "v3base_padded_bf16": Workload("v3base_padded_bf16", 1, "padded", "bf16", 12, 64, 512, 16,
                                   "uniform64"),
    # DeBERTa-v2-xlarge-shaped heavy-padding batch (MNLI-like, ~93 % padding)
    "v2xl_heavypad_fp16": Workload("v2xl_heavypad_fp16", 2, "padded", "fp16", 24, 64, 512, 16,
                                   "lognormal30"),
    # packed varlen, two head shapes
    "packed_varlen_h12d64": Workload("packed_varlen_h12d64", 3, "packed", "bf16", 12, 64, 2048, 64,
                                     "uniform64"),
    "packed_varlen_h6d128": Workload("packed_varlen_h6d128", 3, "packed", "bf16", 6, 128, 2048, 64,
                                     "uniform64"),
    # long-context packed, two head shapes, plus the strict-fp32 case
    "long_packed_h12d64": Workload("long_packed_h12d64", 4, "packed", "bf16", 12, 64, 8192, 16,
                                   "full"),
    "long_packed_h8d128": Workload("long_packed_h8d128", 4, "packed", "bf16", 8, 128, 8192, 16,
                                   "full"),
    "long_packed_fp32": Workload("long_packed_fp32", 4, "packed", "fp32", 12, 64, 2048, 4, "full"),
    # head size 32 (hidden 768 as 24 x 32), packed varlen, bf16
    "packed_varlen_h24d32": Workload("packed_varlen_h24d32", 3, "packed", "bf16", 24, 32, 2048, 64,
                                     "uniform64"),
}


def draw_lengths(w: Workload, rng: np.random.Generator) -> np.ndarray:
    if w.lengths == "full":
        n = np.full(w.batch, w.L, dtype=np.int64)
    elif w.lengths == "first97":
        n = np.full(w.batch, 97, dtype=np.int64)
    elif w.lengths == "uniform64":
        n = rng.integers(64, w.L + 1, size=w.batch, dtype=np.int64)
    elif w.lengths == "lognormal30":
        # median ~30 tokens; sigma 0.65 gives ~93 % padding at B=16, L=512
        raw = rng.lognormal(mean=math.log(30.0), sigma=0.65, size=w.batch)
        n = np.clip(np.round(raw), 8, w.L).astype(np.int64)
    else:
        raise ValueError(w.lengths)
    return n


def _normal(rng, shape, dtype: str, scale: float = 1.0) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x = x * np.float32(scale)
    return torch.from_numpy(x).to(DTYPES[dtype]).contiguous()


@dataclasses.dataclass
class Inputs:
    w: Workload
    lengths: np.ndarray
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    pk: torch.Tensor
    pq: torch.Tensor
    key_mask: Optional[torch.Tensor]   # uint8 [B, L] (padded)
    cu_seqlens: Optional[torch.Tensor]  # int32 [S + 1] (packed)

    @property
    def T(self) -> int:
        return int(self.q.shape[0] * (self.q.shape[1] if self.w.layout == "padded" else 1))

    def seq_slices(self):
        """(start token, length) of every sequence in the flattened token order."""
        if self.w.layout == "packed":
            cu = self.cu_seqlens.numpy()
            return [(int(cu[s]), int(cu[s + 1] - cu[s])) for s in range(cu.size - 1)]
        return [(b * self.w.L, int(n)) for b, n in enumerate(self.lengths)]


def make_inputs(w: Workload | str, *, lengths: Optional[np.ndarray] = None,
                scale: float = 1.0) -> Inputs:
    """Draw one workload.  ``lengths`` overrides the length law (tests);
    ``scale`` multiplies the draws of Q, K, PK and PQ (not V) before the cast,
    so that the logits grow by scale^2 (tests of large score magnitudes)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    rng = np.random.default_rng(w.seed)
    n = draw_lengths(w, rng)
    if lengths is not None:
        n = np.asarray(lengths, dtype=np.int64)
    H, d, P = w.H, w.d, 2 * w.span
    if w.layout == "padded":
        B, L = n.size, w.L
        shape = (B, L, H, d)
        mask = torch.zeros(B, L, dtype=torch.uint8)
        for b in range(B):
            mask[b, : int(n[b])] = 1
        cu = None
    else:
        T = int(n.sum())
        shape = (T, H, d)
        mask = None
        cu = torch.zeros(n.size + 1, dtype=torch.int32)
        cu[1:] = torch.from_numpy(np.cumsum(n).astype(np.int32))
    q = _normal(rng, shape, w.dtype, scale)
    k = _normal(rng, shape, w.dtype, scale)
    v = _normal(rng, shape, w.dtype)
    pk = _normal(rng, (P, H, d), w.dtype, scale)
    pq = _normal(rng, (P, H, d), w.dtype, scale)
    return Inputs(w, n, q, k, v, pk, pq, mask, cu)


def grad_output(x: Inputs, salt: int = 1) -> torch.Tensor:
    """Upstream gradient dL/dO of the backward pass: standard normal values of
    q's shape and dtype, drawn from a generator of its own."""
    rng = np.random.default_rng([x.w.seed, 7919, salt])
    return _normal(rng, tuple(x.q.shape), x.w.dtype)


def custom_inputs(*, layout: str, dtype: str, H: int, d: int, lengths, L: Optional[int] = None,
                  seed: int = 0, buckets: int = 256, max_rel: int = 512,
                  span: Optional[int] = None, scale: float = 1.0) -> Inputs:
    """Same recipe with explicit shapes (edge-case tests); ``scale`` as in
    make_inputs."""
    lengths = np.asarray(lengths, dtype=np.int64)
    if span is None:
        span = buckets if buckets > 0 else max_rel
    if L is None:
        L = int(lengths.max()) if lengths.size else 1
    w = Workload(f"custom_{layout}_{dtype}_H{H}d{d}", seed, layout, dtype, H, d, L,
                 int(lengths.size), "full", buckets, max_rel, span)
    return make_inputs(w, lengths=lengths, scale=scale)
