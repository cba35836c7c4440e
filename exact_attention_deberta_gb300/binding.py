"""Thin ctypes binding of ``include/df_attn.h``: argument marshalling only.

Every step of the attention runs inside ``libdfattn.so``; this module only
turns torch tensors into pointers and sizes, allocates ``out`` / the workspace
with torch when the caller does not pass them, and raises on a non-OK status.
There is no fallback: if the library is missing, importing this module fails.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdfattn.so")

DF_OK, DF_ERR_INVALID_ARG, DF_ERR_UNSUPPORTED, DF_ERR_ALIGNMENT = 0, 1, 2, 3
DF_ERR_WORKSPACE, DF_ERR_CUDA, DF_ERR_DEVICE_TIMEOUT = 4, 5, 6
DF_BF16, DF_FP16, DF_FP32 = 0, 1, 2
_DTYPE = {torch.bfloat16: DF_BF16, torch.float16: DF_FP16, torch.float32: DF_FP32}


class DFError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        super().__init__(f"{what}: {status_string(status)} (status {status})")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run exact_attention_deberta_gb300.build.build() "
                      "(or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)
_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


class _Layout(ctypes.Structure):
    _fields_ = [("header", _sz), ("idx_table", _sz), ("items", _sz), ("scalars", _sz),
                ("keybias", _sz), ("partial", _sz), ("total", _sz), ("max_items", _i),
                ("t_pad", _i), ("table_half", _i), ("diag_pk", _sz), ("diag_pq", _sz),
                ("n_diag", _i), ("diag_m0", _i), ("kaug", _sz), ("kaug_sel", _sz), ("absel", _sz)]


_lib.df_attn_fwd.argtypes = [_vp] * 7 + [_i] * 9 + [_vp, _vp, _sz, _vp]
_lib.df_attn_fwd.restype = _i
_lib.df_attn_plan.argtypes = [_vp] * 6 + [_i] * 9 + [_vp, _vp, _sz, _vp]
_lib.df_attn_plan.restype = _i
_lib.df_attn_workspace_size.argtypes = [_i] * 7
_lib.df_attn_workspace_size.restype = _sz
_lib.df_attn_supported.argtypes = [_i] * 7
_lib.df_attn_supported.restype = _i
_lib.df_attn_status_string.argtypes = [_i]
_lib.df_attn_status_string.restype = ctypes.c_char_p
_lib.df_attn_get_device_status.argtypes = [_vp, _vp]
_lib.df_attn_get_device_status.restype = _i
_lib.df_rel_index_table.argtypes = [_i, _i, _i, _i, _vp, _vp]
_lib.df_rel_index_table.restype = _i
_lib.df_attn_workspace_layout.argtypes = [_i] * 7 + [ctypes.POINTER(_Layout)]
_lib.df_attn_workspace_layout.restype = _i
_lib.df_attn_set_profile_events.argtypes = [_vp, _vp]
_lib.df_attn_set_profile_events.restype = None
_lib.df_attn_set_profile_split.argtypes = [_vp]
_lib.df_attn_set_profile_split.restype = None
_lib.df_attn_set_wait_budget.argtypes = [ctypes.c_ulonglong]
_lib.df_attn_set_wait_budget.restype = None
_lib.df_attn_last_launch_count.argtypes = []
_lib.df_attn_last_launch_count.restype = _i


def status_string(status: int) -> str:
    return _lib.df_attn_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != DF_OK:
        raise DFError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def default_span(buckets: int, max_rel: int) -> int:
    """DeBERTa's attention span: position_buckets if bucketing is on, else max_rel."""
    return buckets if buckets > 0 else max_rel


def df_attn_workspace_size(B, H, L, d, buckets=256, max_rel=512, span=None) -> int:
    span = default_span(buckets, max_rel) if span is None else span
    return int(_lib.df_attn_workspace_size(B, H, L, d, buckets, max_rel, span))


def df_attn_supported(H, L, d, dtype, buckets=256, max_rel=512, span=None) -> int:
    span = default_span(buckets, max_rel) if span is None else span
    dt = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(_lib.df_attn_supported(H, L, d, dt, buckets, max_rel, span))


def df_attn_workspace_layout(B, H, L, d, buckets=256, max_rel=512, span=None) -> dict:
    span = default_span(buckets, max_rel) if span is None else span
    lay = _Layout()
    _check(_lib.df_attn_workspace_layout(B, H, L, d, buckets, max_rel, span, ctypes.byref(lay)),
           "df_attn_workspace_layout")
    return {name: getattr(lay, name) for name, _ in _Layout._fields_}


def _shape_args(q, key_mask, cu_seqlens, max_seqlen):
    if (key_mask is None) == (cu_seqlens is None):
        raise ValueError("pass exactly one of key_mask (padded) and cu_seqlens (packed)")
    if key_mask is not None:
        B, L, H, d = q.shape
        return B, H, L, B * L, d
    T, H, d = q.shape
    B = cu_seqlens.numel() - 1
    if max_seqlen is None:
        raise ValueError("packed mode needs max_seqlen (an upper bound of every length)")
    return B, H, int(max_seqlen), T, d


def _prepare(q, k, v, pos_key, pos_query, key_mask, cu_seqlens, max_seqlen, buckets, max_rel,
             span, out, workspace):
    B, H, L, T, d = _shape_args(q, key_mask, cu_seqlens, max_seqlen)
    span = default_span(buckets, max_rel) if span is None else span
    for name, t in (("q", q), ("k", k), ("v", v), ("pos_key", pos_key), ("pos_query", pos_query)):
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if t.dtype != q.dtype:
            raise ValueError(f"{name} dtype {t.dtype} != q dtype {q.dtype}")
    if q.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if key_mask is not None and (key_mask.dtype != torch.uint8 or not key_mask.is_contiguous()):
        raise ValueError("key_mask must be a contiguous uint8 tensor")
    if cu_seqlens is not None and (cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_contiguous()):
        raise ValueError("cu_seqlens must be a contiguous int32 tensor")
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        size = df_attn_workspace_size(B, H, L, d, buckets, max_rel, span)
        workspace = torch.empty(max(size, 256), dtype=torch.uint8, device=q.device)
    return B, H, L, T, d, span, out, workspace


def df_attn_fwd(q, k, v, pos_key, pos_query, key_mask=None, cu_seqlens=None, *, max_seqlen=None,
                buckets=256, max_rel=512, span=None, out=None, workspace=None, stream=None):
    """Fused disentangled-attention forward; returns ``out`` (same layout as q)."""
    B, H, L, T, d, span, out, workspace = _prepare(q, k, v, pos_key, pos_query, key_mask,
                                                   cu_seqlens, max_seqlen, buckets, max_rel,
                                                   span, out, workspace)
    st = _lib.df_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(pos_key), _ptr(pos_query),
                          _ptr(key_mask), _ptr(cu_seqlens), B, H, L, T, d, buckets, max_rel,
                          span, _DTYPE[q.dtype], _ptr(out), _ptr(workspace),
                          workspace.numel(), _stream(stream))
    _check(st, "df_attn_fwd")
    return out


_lib.df_attn_fwd_fp32_fast.argtypes = [_vp] * 7 + [_i] * 8 + [_vp, _vp, _sz, _vp]
_lib.df_attn_fwd_fp32_fast.restype = _i
_lib.df_attn_fwd_fp32_fast_workspace_size.argtypes = [_i] * 7
_lib.df_attn_fwd_fp32_fast_workspace_size.restype = _sz


def df_attn_fwd_fp32_fast_workspace_size(B, H, L, d, buckets=256, max_rel=512, span=None) -> int:
    span = default_span(buckets, max_rel) if span is None else span
    return int(_lib.df_attn_fwd_fp32_fast_workspace_size(B, H, L, d, buckets, max_rel, span))


def df_attn_fwd_fp32_fast(q, k, v, pos_key, pos_query, key_mask=None, cu_seqlens=None, *,
                          max_seqlen=None, buckets=256, max_rel=512, span=None, out=None,
                          workspace=None, stream=None):
    """Fast fp32 mode: fp32 tensors, computed on the fp16 tensor-core path
    (inputs rounded to fp16, |x| <= 65504); returns ``out`` (fp32)."""
    if q.dtype != torch.float32:
        raise ValueError("df_attn_fwd_fp32_fast takes float32 tensors")
    if not q.is_cuda:
        raise ValueError("q must be a contiguous CUDA tensor")
    B, H, L, T, d = _shape_args(q, key_mask, cu_seqlens, max_seqlen)
    span = default_span(buckets, max_rel) if span is None else span
    if workspace is None:
        size = df_attn_fwd_fp32_fast_workspace_size(B, H, L, d, buckets, max_rel, span)
        workspace = torch.empty(max(size, 256), dtype=torch.uint8, device=q.device)
    B, H, L, T, d, span, out, workspace = _prepare(q, k, v, pos_key, pos_query, key_mask,
                                                   cu_seqlens, max_seqlen, buckets, max_rel,
                                                   span, out, workspace)
    st = _lib.df_attn_fwd_fp32_fast(_ptr(q), _ptr(k), _ptr(v), _ptr(pos_key), _ptr(pos_query),
                                    _ptr(key_mask), _ptr(cu_seqlens), B, H, L, T, d, buckets,
                                    max_rel, span, _ptr(out), _ptr(workspace), workspace.numel(),
                                    _stream(stream))
    _check(st, "df_attn_fwd_fp32_fast")
    return out


_lib.df_attn_bwd.argtypes = [_vp] * 8 + [_i] * 9 + [_vp] * 5 + [_vp, _sz, _vp]
_lib.df_attn_bwd.restype = _i
_lib.df_attn_bwd_workspace_size.argtypes = [_i] * 7
_lib.df_attn_bwd_workspace_size.restype = _sz


def df_attn_bwd_workspace_size(B, H, L, d, buckets=256, max_rel=512, span=None) -> int:
    span = default_span(buckets, max_rel) if span is None else span
    return int(_lib.df_attn_bwd_workspace_size(B, H, L, d, buckets, max_rel, span))


def df_attn_bwd(q, k, v, pos_key, pos_query, dout, key_mask=None, cu_seqlens=None, *,
                max_seqlen=None, buckets=256, max_rel=512, span=None, grads=None,
                workspace=None, stream=None):
    """Backward pass; returns float32 (dq, dk, dv, dpos_key, dpos_query).

    ``grads`` may pass those five tensors preallocated (float32, contiguous)."""
    placeholder = workspace if workspace is not None else q  # checked, not used
    B, H, L, T, d, span, _, _ = _prepare(q, k, v, pos_key, pos_query, key_mask, cu_seqlens,
                                         max_seqlen, buckets, max_rel, span, q, placeholder)
    if workspace is None:
        size = df_attn_bwd_workspace_size(B, H, L, d, buckets, max_rel, span)
        if size == 0:
            _check(DF_ERR_UNSUPPORTED, "df_attn_bwd_workspace_size")
        workspace = torch.empty(size, dtype=torch.uint8, device=q.device)
    if dout.shape != q.shape or dout.dtype != q.dtype or not dout.is_contiguous():
        raise ValueError("dout must match q in shape and dtype and be contiguous")
    if grads is None:
        f32 = dict(dtype=torch.float32, device=q.device)
        grads = (torch.empty(q.shape, **f32), torch.empty(q.shape, **f32), torch.empty(q.shape, **f32),
                 torch.empty(pos_key.shape, **f32), torch.empty(pos_key.shape, **f32))
    dq, dk, dv, dpk, dpq = grads
    st = _lib.df_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(pos_key), _ptr(pos_query), _ptr(dout),
                          _ptr(key_mask), _ptr(cu_seqlens), B, H, L, T, d, buckets, max_rel, span,
                          _DTYPE[q.dtype], _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dpk), _ptr(dpq),
                          _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "df_attn_bwd")
    return dq, dk, dv, dpk, dpq


_ll = ctypes.c_longlong
_lib.df_attn_fwd_host.argtypes = [_vp] * 7 + [_i] * 9 + [_vp, _ll, _vp, _sz, _vp]
_lib.df_attn_fwd_host.restype = _i
_lib.df_attn_fwd_host_scratch_size.argtypes = [_i] * 8 + [_ll]
_lib.df_attn_fwd_host_scratch_size.restype = _sz


def df_attn_fwd_host_scratch_size(B, H, L, d, dtype, buckets=256, max_rel=512, span=None,
                                  group_tokens=0) -> int:
    span = default_span(buckets, max_rel) if span is None else span
    dt = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(_lib.df_attn_fwd_host_scratch_size(B, H, L, d, buckets, max_rel, span, dt, group_tokens))


def df_attn_fwd_host(q, k, v, pos_key, pos_query, key_mask=None, cu_seqlens=None, *, max_seqlen=None,
                     buckets=256, max_rel=512, span=None, out=None, group_tokens=0, scratch=None,
                     stream=None):
    """Forward from host (CPU, ideally pinned) tensors with the copies overlapped
    with the kernels; returns ``out`` (a host tensor), complete once ``stream``
    is synchronised."""
    B, H, L, T, d = _shape_args(q, key_mask, cu_seqlens, max_seqlen)
    span = default_span(buckets, max_rel) if span is None else span
    for name, t in (("q", q), ("k", k), ("v", v), ("pos_key", pos_key), ("pos_query", pos_query),
                    ("key_mask", key_mask), ("cu_seqlens", cu_seqlens), ("out", out)):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous host tensor")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if scratch is None:
        size = df_attn_fwd_host_scratch_size(B, H, L, d, q.dtype, buckets, max_rel, span, group_tokens)
        if size == 0:
            _check(DF_ERR_UNSUPPORTED, "df_attn_fwd_host_scratch_size")
        scratch = torch.empty(size, dtype=torch.uint8, device="cuda")
    st = _lib.df_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(pos_key), _ptr(pos_query), _ptr(key_mask),
                               _ptr(cu_seqlens), B, H, L, T, d, buckets, max_rel, span, _DTYPE[q.dtype],
                               _ptr(out), int(group_tokens), _ptr(scratch), scratch.numel(),
                               _stream(stream))
    _check(st, "df_attn_fwd_host")
    return out


def df_attn_plan(q, k, pos_key, pos_query, key_mask=None, cu_seqlens=None, *, max_seqlen=None,
                 buckets=256, max_rel=512, span=None, out=None, workspace=None, stream=None):
    """Planning step alone; returns (out, workspace)."""
    B, H, L, T, d, span, out, workspace = _prepare(q, k, None, pos_key, pos_query, key_mask,
                                                   cu_seqlens, max_seqlen, buckets, max_rel,
                                                   span, out, workspace)
    st = _lib.df_attn_plan(_ptr(q), _ptr(k), _ptr(pos_key), _ptr(pos_query), _ptr(key_mask),
                           _ptr(cu_seqlens), B, H, L, T, d, buckets, max_rel, span,
                           _DTYPE[q.dtype], _ptr(out), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    _check(st, "df_attn_plan")
    return out, workspace


_lib.df_attn_fwd_noalloc.argtypes = [_vp] * 7 + [_i] * 9 + [_vp, _vp]
_lib.df_attn_fwd_noalloc.restype = _i
NOALLOC_SCRATCH_BYTES = 64 << 20


def df_attn_fwd_noalloc(q, k, v, pos_key, pos_query, key_mask=None, cu_seqlens=None, *, out,
                        max_seqlen=None, buckets=256, max_rel=512, span=None, stream=None):
    """df_attn_fwd for callers that cannot allocate device memory: the library's
    built-in scratch array replaces the workspace, and ``out`` must be provided."""
    B, H, L, T, d = _shape_args(q, key_mask, cu_seqlens, max_seqlen)
    span = default_span(buckets, max_rel) if span is None else span
    st = _lib.df_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(pos_key), _ptr(pos_query),
                                  _ptr(key_mask), _ptr(cu_seqlens), B, H, L, T, d, buckets,
                                  max_rel, span, _DTYPE[q.dtype], _ptr(out), _stream(stream))
    _check(st, "df_attn_fwd_noalloc")
    return out


_lib.df_attn_noalloc_get_device_status.argtypes = [_vp]
_lib.df_attn_noalloc_get_device_status.restype = _i


def df_attn_noalloc_get_device_status(stream=None) -> int:
    """Status word of the latest df_attn_fwd_noalloc call on the current device
    (read and cleared; synchronises the stream)."""
    return int(_lib.df_attn_noalloc_get_device_status(_stream(stream)))


def df_attn_get_device_status(workspace, stream=None) -> int:
    return int(_lib.df_attn_get_device_status(_ptr(workspace), _stream(stream)))


def df_rel_index_table(buckets, max_rel, span, max_len, out=None, stream=None, device="cuda"):
    if out is None:
        out = torch.empty(2 * max_len - 1, dtype=torch.int32, device=device)
    _check(_lib.df_rel_index_table(buckets, max_rel, span, max_len, _ptr(out), _stream(stream)),
           "df_rel_index_table")
    return out


def df_attn_set_profile_events(start=None, stop=None):
    h = lambda e: None if e is None else ctypes.c_void_p(e.cuda_event)  # noqa: E731
    _lib.df_attn_set_profile_events(h(start), h(stop))


def df_attn_set_profile_split(mid=None):
    _lib.df_attn_set_profile_split(None if mid is None else ctypes.c_void_p(mid.cuda_event))


def df_attn_set_wait_budget(cycles: int):
    _lib.df_attn_set_wait_budget(int(cycles))


def df_attn_last_launch_count() -> int:
    return int(_lib.df_attn_last_launch_count())


_lib.df_pack_info.argtypes = [_vp, _i, _i, _vp, _vp, _vp, _vp, _vp]
_lib.df_pack_info.restype = _i
_lib.df_pack_rows.argtypes = [_vp, _vp, _vp, _i, _sz, _vp, _vp]
_lib.df_pack_rows.restype = _i
_lib.df_unpack_rows.argtypes = [_vp, _vp, _i, _sz, _vp, _vp]
_lib.df_unpack_rows.restype = _i


class PackedInfo:
    """Metadata of a padded -> packed conversion, reusable across layers: the
    packed -> padded row list, its inverse (-1 at padding), cu_seqlens, the
    token count and the longest sequence."""

    def __init__(self, batch, seqlen, cu_seqlens, indices, inverse, stats, total, max_seqlen):
        self.batch, self.seqlen = batch, seqlen
        self.cu_seqlens, self.indices, self.inverse = cu_seqlens, indices, inverse
        self.stats = stats  # device int32 {T, max_seqlen}
        self.total, self.max_seqlen = total, max_seqlen


def df_pack_info(mask, stream=None) -> PackedInfo:
    """Metadata of a uint8 mask [B, L] (nonzero = valid).  Reads T and
    max_seqlen back to the host (one synchronisation of the stream)."""
    if not mask.is_cuda or mask.dtype != torch.uint8 or mask.dim() != 2 or not mask.is_contiguous():
        raise ValueError("mask must be a contiguous CUDA uint8 tensor [B, L]")
    B, L = mask.shape
    dev = mask.device
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
    indices = torch.empty(B * L, dtype=torch.int32, device=dev)
    inverse = torch.empty(B * L, dtype=torch.int32, device=dev)
    stats = torch.empty(2, dtype=torch.int32, device=dev)
    _check(_lib.df_pack_info(_ptr(mask), B, L, _ptr(cu), _ptr(indices), _ptr(inverse), _ptr(stats),
                             _stream(stream)), "df_pack_info")
    total, max_seqlen = (int(v) for v in stats.cpu())
    return PackedInfo(B, L, cu, indices[:total], inverse, stats, total, max_seqlen)


def _row_bytes(t, lead):
    return t[0].numel() * t.element_size() if lead == 1 else t[0, 0].numel() * t.element_size()


def pack_padded_with_info(hidden_states, attention_mask, stream=None):
    """[B, L, ...] -> ([T, ...] rows, cu_seqlens, PackedInfo)."""
    if not hidden_states.is_cuda or not hidden_states.is_contiguous():
        raise ValueError("hidden_states must be a contiguous CUDA tensor [B, L, ...]")
    mask = attention_mask.to(torch.uint8).contiguous()
    info = df_pack_info(mask, stream)
    B, L = info.batch, info.seqlen
    if tuple(hidden_states.shape[:2]) != (B, L):
        raise ValueError("hidden_states and attention_mask disagree on [B, L]")
    tokens = torch.empty((max(info.total, 1),) + tuple(hidden_states.shape[2:]), dtype=hidden_states.dtype,
                         device=hidden_states.device)
    if info.total > 0:
        _check(_lib.df_pack_rows(_ptr(hidden_states), _ptr(info.indices), _ptr(info.stats), B * L,
                                 _row_bytes(hidden_states, 2), _ptr(tokens), _stream(stream)),
               "df_pack_rows")
    return tokens[:info.total], info.cu_seqlens, info


def unpack_packed(packed, cu_seqlens, seqlen, packed_info, stream=None):
    """[T, ...] -> ([B, L, ...] with zeros at padding, the padded-row mask)."""
    info = packed_info
    if seqlen != info.seqlen:
        raise ValueError("seqlen differs from the metadata's")
    if not packed.is_cuda or not packed.is_contiguous() or packed.shape[0] != info.total:
        raise ValueError("packed must be a contiguous CUDA tensor with the metadata's token count")
    B, L = info.batch, info.seqlen
    out = torch.empty((B, L) + tuple(packed.shape[1:]), dtype=packed.dtype, device=packed.device)
    src = packed if info.total > 0 else torch.zeros((1,) + tuple(packed.shape[1:]), dtype=packed.dtype,
                                                    device=packed.device)
    _check(_lib.df_unpack_rows(_ptr(src), _ptr(info.inverse), B * L, _row_bytes(out, 2), _ptr(out),
                               _stream(stream)), "df_unpack_rows")
    return out, (info.inverse >= 0).view(B, L)


_PP = ctypes.POINTER(ctypes.c_void_p)
_lib.df_linear.argtypes = [_vp, _i, _i, _i, _PP, _PP, _i, _PP, _i, _i, _vp, _vp]
_lib.df_linear.restype = _i


def _ptr_array(ts):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = None if t is None else t.data_ptr()
    return arr


LINEAR_NONE, LINEAR_GELU = 0, 1


def df_linear(x, weights, biases=None, outs=None, status=None, stream=None, activation=LINEAR_NONE):
    """[act(x . W_i^T + b_i)] for 1..3 weights W_i [N, K] (nn.Linear layout) sharing x [M, K]."""
    if x.dim() != 2 or not x.is_cuda or not x.is_contiguous() or x.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("x must be a contiguous CUDA bf16/fp16 matrix [M, K]")
    M, K = x.shape
    N = weights[0].shape[0]
    for w in weights:
        if tuple(w.shape) != (N, K) or w.dtype != x.dtype or not w.is_contiguous() or not w.is_cuda:
            raise ValueError("every weight must be a contiguous CUDA [N, K] matrix of x's dtype")
    if biases is not None:
        for b in biases:
            if b is not None and (b.shape != (N,) or b.dtype != x.dtype or not b.is_contiguous()):
                raise ValueError("biases must be [N] vectors of x's dtype")
    if outs is None:
        outs = [torch.empty(M, N, dtype=x.dtype, device=x.device) for _ in weights]
    st = _lib.df_linear(_ptr(x), M, K, len(weights), _ptr_array(weights),
                        _ptr_array(biases) if biases is not None else None, N, _ptr_array(outs),
                        int(activation), _DTYPE[x.dtype], _ptr(status), _stream(stream))
    _check(st, "df_linear")
    return outs


def qkv_projection(hidden, w_qkv, b_qkv, heads, stream=None):
    """Fused QKV projection: hidden [T, hidden] with the stacked weight [3 H d, hidden]
    (and bias [3 H d]) -> q, k, v, each [T, H, d]."""
    n3 = w_qkv.shape[0]
    n = n3 // 3
    ws = [w_qkv[i * n:(i + 1) * n] for i in range(3)]
    bs = None if b_qkv is None else [b_qkv[i * n:(i + 1) * n] for i in range(3)]
    outs = df_linear(hidden, ws, bs, stream=stream)
    T = hidden.shape[0]
    return [o.view(T, heads, n // heads) for o in outs]


def rel_projection(rel_embeddings, w_key, b_key, w_query, b_query, heads, stream=None):
    """PK = rel . W_k^T + b_k and PQ = rel . W_q^T + b_q, each [2 span, H, d]."""
    outs = df_linear(rel_embeddings, [w_key, w_query], [b_key, b_query], stream=stream)
    R, n = outs[0].shape
    return [o.view(R, heads, n // heads) for o in outs]


_lib.df_layernorm.argtypes = [_vp, _vp, _vp, _vp, _i, _i, ctypes.c_float, _vp, _i, _vp]
_lib.df_layernorm.restype = _i


def df_layernorm(x, gamma, beta, residual=None, eps=1e-7, out=None, stream=None):
    """LayerNorm(x + residual) * gamma + beta over the last dimension of [M, N]."""
    M, N = x.shape
    if out is None:
        out = torch.empty_like(x)
    _check(_lib.df_layernorm(_ptr(x), _ptr(residual), _ptr(gamma), _ptr(beta), M, N, float(eps), _ptr(out),
                             _DTYPE[x.dtype], _stream(stream)), "df_layernorm")
    return out


raw_library = _lib
