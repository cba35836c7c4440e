"""Failure detection on the GPU without a fault: a wait budget far below the
latency of any copy makes the kernels' bounded mbarrier waits run out.  The
kernels record DF_ERR_DEVICE_TIMEOUT in the workspace header, drain their own
copies and MMAs in flight, free their tensor memory and return; the context
stays usable and the next call with the default budget is exact again."""

import pytest
import torch

from exact_attention_deberta_gb300 import synth

from _parity import assert_close, oracle_full, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout,dtype,d", [("packed", "bf16", 64), ("padded", "fp16", 64),
                                            ("packed", "bf16", 128)])
def test_wait_budget_runs_out_and_recovers(lib, layout, dtype, d):
    x = synth.custom_inputs(layout=layout, dtype=dtype, H=2, d=d, lengths=[700, 300], L=700, seed=9)
    B = len(x.lengths)
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    ws = torch.empty(lib.df_attn_workspace_size(B, x.w.H, x.w.L, x.w.d, **kw), dtype=torch.uint8,
                     device="cuda")
    lib.df_attn_set_wait_budget(1)
    try:
        run_gpu(lib, x, workspace=ws)
        st = lib.df_attn_get_device_status(ws)
    finally:
        lib.df_attn_set_wait_budget(0)
    assert st == lib.DF_ERR_DEVICE_TIMEOUT, lib.status_string(st)
    # the context is still usable and the default budget gives exact results again
    out = run_gpu(lib, x)
    assert_close(out.double().cpu().numpy(), oracle_full(x), dtype, "after timeout")
