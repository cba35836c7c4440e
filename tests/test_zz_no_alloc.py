"""df_attn_fwd_noalloc, the entry point for callers that cannot allocate device
memory (for example a plug-in whose host application owns all device memory and
offers it no allocator, or a service that forbids cudaMalloc / cudaFree once it
is running).  Both entry points run the same deterministic kernels, so its
output must equal df_attn_fwd's (caller-provided workspace) bit for bit, on
consecutive calls that share the built-in scratch; errors raised on the device
must be readable through df_attn_noalloc_get_device_status.

Kept in a file of its own that pytest collects last."""

import pytest
import torch

from exact_attention_deberta_gb300 import synth

from _parity import run_gpu

pytestmark = pytest.mark.gpu


CASES = {
    "padded_bf16": lambda: synth.make_inputs("v3base_padded_bf16"),
    "packed_bf16_d128": lambda: synth.custom_inputs(layout="packed", dtype="bf16", H=4, d=128,
                                                    lengths=[1500, 3, 800], seed=12),
    "packed_fp16_far": lambda: synth.custom_inputs(layout="packed", dtype="fp16", H=2, d=64,
                                                   lengths=[2500, 64], seed=13),
    "padded_fp32": lambda: synth.make_inputs("tiny_fp32_pad97"),
}


def _dev(x):
    return {n: None if getattr(x, n) is None else getattr(x, n).cuda()
            for n in ("q", "k", "v", "pk", "pq", "key_mask", "cu_seqlens")}


def _noalloc(lib, x, dev, out):
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    if x.w.layout == "padded":
        lib.df_attn_fwd_noalloc(dev["q"], dev["k"], dev["v"], dev["pk"], dev["pq"],
                                key_mask=dev["key_mask"], out=out, **kw)
    else:
        lib.df_attn_fwd_noalloc(dev["q"], dev["k"], dev["v"], dev["pk"], dev["pq"],
                                cu_seqlens=dev["cu_seqlens"], max_seqlen=x.w.L, out=out, **kw)


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_workspace_entry_point(lib, name):
    x = CASES[name]()
    B = x.q.shape[0] if x.w.layout == "padded" else x.cu_seqlens.numel() - 1
    assert lib.df_attn_workspace_size(B, x.w.H, x.w.L, x.w.d) <= lib.NOALLOC_SCRATCH_BYTES
    dev = _dev(x)
    ref = run_gpu(lib, x, dev_inputs=dev)
    torch.cuda.synchronize()
    for call in range(2):  # the second call reuses the scratch the first one left behind
        out = torch.full_like(dev["q"], float("nan"))
        _noalloc(lib, x, dev, out)
        st = lib.df_attn_noalloc_get_device_status()
        assert st == lib.DF_OK, f"call {call}: {lib.status_string(st)}"
        assert torch.equal(out, ref), f"call {call}: differs from df_attn_fwd"


def test_noalloc_reports_device_errors(lib):
    # a wait budget of one cycle makes the kernels' bounded waits run out (no
    # fault: they record the timeout, drain their copies and return)
    x = CASES["packed_fp16_far"]()
    dev = _dev(x)
    out = torch.empty_like(dev["q"])
    lib.df_attn_set_wait_budget(1)
    try:
        _noalloc(lib, x, dev, out)
        st = lib.df_attn_noalloc_get_device_status()
    finally:
        lib.df_attn_set_wait_budget(0)
    assert st == lib.DF_ERR_DEVICE_TIMEOUT, lib.status_string(st)
    assert lib.df_attn_noalloc_get_device_status() == lib.DF_OK  # read clears it
    ref = run_gpu(lib, x, dev_inputs=dev)
    _noalloc(lib, x, dev, out)
    assert lib.df_attn_noalloc_get_device_status() == lib.DF_OK
    assert torch.equal(out, ref)


def test_noalloc_rejects_problems_beyond_the_scratch(lib):
    x = synth.custom_inputs(layout="packed", dtype="bf16", H=12, d=64, lengths=[64], L=64, seed=1)
    need = lib.df_attn_workspace_size(64, 12, 8192, 64)
    assert need > lib.NOALLOC_SCRATCH_BYTES
    out = torch.empty_like(x.q).cuda()
    with pytest.raises(lib.DFError) as err:
        lib.df_attn_fwd_noalloc(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.pk.cuda(), x.pq.cuda(),
                                cu_seqlens=torch.tensor([0] + [1] * 64, dtype=torch.int32).cuda(),
                                max_seqlen=8192, out=out)
    assert err.value.status == lib.DF_ERR_WORKSPACE
