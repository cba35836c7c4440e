"""Host-buffer forward (df_attn_fwd_host): groups of whole sequences with the
copies overlapped must give exactly the bytes of one df_attn_fwd call on the
whole batch (the same kernels on independent sequences), for pinned and
pageable buffers, packed and padded layouts, and group sizes that force many
groups, groups of one sequence and empty sequences."""

import pytest
import torch

from exact_attention_deberta_gb300 import synth

pytestmark = pytest.mark.gpu


def _device_out(lib, x):
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    d = [getattr(x, n).cuda() for n in ("q", "k", "v", "pk", "pq")]
    if x.w.layout == "padded":
        o = lib.df_attn_fwd(*d, key_mask=x.key_mask.cuda(), **kw)
    else:
        o = lib.df_attn_fwd(*d, cu_seqlens=x.cu_seqlens.cuda(), max_seqlen=x.w.L, **kw)
    torch.cuda.synchronize()
    return o.cpu()


def _host_out(lib, x, group_tokens, pinned):
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    h = [getattr(x, n).contiguous() for n in ("q", "k", "v", "pk", "pq")]
    if pinned:
        h = [t.pin_memory() for t in h]
    out = torch.full(x.q.shape, float("nan"), dtype=x.q.dtype)
    if pinned:
        out = out.pin_memory()
    if x.w.layout == "padded":
        lib.df_attn_fwd_host(*h, key_mask=x.key_mask, out=out, group_tokens=group_tokens, **kw)
    else:
        lib.df_attn_fwd_host(*h, cu_seqlens=x.cu_seqlens, max_seqlen=x.w.L, out=out,
                             group_tokens=group_tokens, **kw)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("group_tokens", [0, 1, 900])
def test_host_forward_packed_is_bit_exact(lib, group_tokens, pinned):
    x = synth.custom_inputs(layout="packed", dtype="bf16", H=3, d=64, lengths=[300, 0, 77, 512, 1, 260],
                            seed=9)
    ref = _device_out(lib, x)
    got = _host_out(lib, x, group_tokens, pinned)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("group_tokens", [0, 200])
def test_host_forward_padded_is_bit_exact(lib, group_tokens):
    x = synth.custom_inputs(layout="padded", dtype="fp16", H=2, d=128, lengths=[100, 37, 150, 64, 1],
                            L=150, seed=10)
    ref = _device_out(lib, x)
    got = _host_out(lib, x, group_tokens, True)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_host_forward_long_workload_groups(lib):
    x = synth.make_inputs("long_packed_h12d64")
    ref = _device_out(lib, x)
    got = _host_out(lib, x, 16384, True)   # eight groups of two 8192-token sequences
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_host_forward_head_size_32(lib):
    """Head size 32 runs the d = 64 kernels on widened copies: the host-buffer
    path must give the same bytes as the device call there too."""
    x = synth.custom_inputs(layout="packed", dtype="bf16", H=4, d=32, lengths=[700, 1, 129, 0, 300], seed=11)
    ref = _device_out(lib, x)
    got = _host_out(lib, x, 0, True)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
