"""Fast fp32 mode (df_attn_fwd_fp32_fast): fp32 tensors computed on the fp16
tensor-core path, against the float64 oracle on the original fp32 inputs.

Tolerance: the fp16 path's bound (max-abs 1e-2, rel-L2 3e-3) covers the
rounding of P and of the output to fp16; here the inputs are rounded to fp16
as well (relative 2^-11 each), which moves a score by about 1e-3 for N(0, 1)
data at d = 64 (three dot products of d terms with independent rounding
errors, scaled by 1/sqrt(3 d)) -- an error of the same size as the output
rounding, hence 1.5 times the fp16 bound."""

import numpy as np
import pytest
import torch

from exact_attention_deberta_gb300 import synth
from _parity import errors, oracle_full

pytestmark = pytest.mark.gpu

TOL_FAST32 = (1.5e-2, 4.5e-3)

CASES = [
    # far tiles (distances past the saturation point), a one-token sequence
    dict(layout="packed", H=2, d=64, lengths=[700, 130, 1], L=700, seed=11),
    dict(layout="padded", H=2, d=128, lengths=[77, 300], L=300, seed=12),
    dict(layout="packed", H=3, d=128, lengths=[600, 257], L=600, seed=13),
    dict(layout="packed", H=4, d=32, lengths=[300, 64], L=300, seed=14),
]


def _run(lib, x, workspace=None):
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    d = [getattr(x, n).cuda() for n in ("q", "k", "v", "pk", "pq")]
    if x.w.layout == "padded":
        o = lib.df_attn_fwd_fp32_fast(*d, key_mask=x.key_mask.cuda(), workspace=workspace, **kw)
    else:
        o = lib.df_attn_fwd_fp32_fast(*d, cu_seqlens=x.cu_seqlens.cuda(), max_seqlen=x.w.L,
                                      workspace=workspace, **kw)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c['layout']}-d{c['d']}-L{c['L']}")
def test_fast_fp32_matches_oracle(lib, case):
    x = synth.custom_inputs(dtype="fp32", **case)
    assert x.q.dtype == torch.float32
    B = x.key_mask.shape[0] if x.w.layout == "padded" else x.cu_seqlens.numel() - 1
    size = lib.df_attn_fwd_fp32_fast_workspace_size(B, x.w.H, x.w.L, x.w.d, x.w.buckets,
                                                    x.w.max_rel, x.w.span)
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    got = _run(lib, x, ws)
    assert got.dtype == torch.float32
    assert lib.df_attn_get_device_status(ws) == lib.DF_OK
    # the conversions plus the fp16 forward's own launches
    assert lib.df_attn_last_launch_count() >= 4
    ref = oracle_full(x)
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g))
    max_abs, rel = errors(g, ref)
    assert max_abs <= TOL_FAST32[0] and rel <= TOL_FAST32[1], (max_abs, rel)
    # padded query rows are exact zeros
    if x.w.layout == "padded":
        pad = ~x.key_mask.bool()
        assert torch.all(got.cpu()[pad] == 0)


def test_fast_fp32_reports_values_out_of_fp16_range(lib):
    x = synth.custom_inputs(layout="packed", dtype="fp32", H=2, d=64, lengths=[200], L=200, seed=15)
    x.k[17, 1, 5] = 1.0e5  # beyond fp16's largest finite value
    size = lib.df_attn_fwd_fp32_fast_workspace_size(1, 2, 200, 64, x.w.buckets, x.w.max_rel, x.w.span)
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    _run(lib, x, ws)
    assert lib.df_attn_get_device_status(ws) == lib.DF_ERR_INVALID_ARG
    assert lib.df_attn_get_device_status(ws) == lib.DF_OK  # the read clears it
    # a clean call on the same workspace reports nothing
    x.k[17, 1, 5] = 0.5
    _run(lib, x, ws)
    assert lib.df_attn_get_device_status(ws) == lib.DF_OK
