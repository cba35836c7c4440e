"""The C-ABI library loads, exports every entry point of include/df_attn.h, and
rejects out-of-contract arguments on the host (no GPU needed: every call here
returns before its first CUDA call)."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "df_attn.h")


@pytest.fixture(scope="module")
def binding():
    from exact_attention_deberta_gb300.build import build
    build()
    from exact_attention_deberta_gb300 import binding as b
    return b


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(df_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("df_attn_fwd", "df_attn_workspace_size", "df_attn_supported",
                 "df_attn_status_string", "df_attn_get_device_status", "df_rel_index_table"):
        assert must in names


def test_every_declared_symbol_is_exported(binding):
    lib = ctypes.CDLL(binding.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(binding):
    for s in range(7):
        assert binding.status_string(s) and binding.status_string(s) != "unknown status"
    assert binding.status_string(99) == "unknown status"


def test_supported_matrix(binding):
    import torch
    ok = binding.DF_OK
    assert binding.df_attn_supported(12, 8192, 64, torch.bfloat16) == ok
    assert binding.df_attn_supported(8, 8192, 128, torch.float16) == ok
    assert binding.df_attn_supported(12, 2048, 64, torch.float32) == ok
    assert binding.df_attn_supported(12, 512, 48, torch.bfloat16) == binding.DF_ERR_UNSUPPORTED
    assert binding.df_attn_supported(12, 512, 32, torch.bfloat16) == ok
    assert binding.df_attn_supported(12, 512, 96, torch.bfloat16) == binding.DF_ERR_UNSUPPORTED
    assert binding.df_attn_supported(0, 512, 64, torch.bfloat16) == binding.DF_ERR_INVALID_ARG
    assert binding.df_attn_supported(12, 0, 64, torch.bfloat16) == binding.DF_ERR_INVALID_ARG
    # buckets/2 must stay below max_rel - 1 for the logarithm to grow
    assert binding.df_attn_supported(12, 512, 64, torch.bfloat16, buckets=1024, max_rel=512,
                                     span=1024) == binding.DF_ERR_INVALID_ARG
    assert binding.df_attn_supported(12, 512, 64, 7) == binding.DF_ERR_INVALID_ARG


def test_workspace_size_and_layout(binding):
    size = binding.df_attn_workspace_size(16, 12, 8192, 64)
    lay = binding.df_attn_workspace_layout(16, 12, 8192, 64)
    assert size == lay["total"] > 0
    offs = [lay[k] for k in ("header", "idx_table", "items", "scalars", "keybias", "partial")]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lay["max_items"] == 16 * 12 * 64
    assert lay["table_half"] == 8192 + 128
    assert binding.df_attn_workspace_size(16, 12, 8192, 48) == 0


@pytest.mark.parametrize("buckets,max_rel,span,L", [
    (256, 512, 256, 8192), (256, 512, 256, 300), (0, 512, 512, 2048), (64, 128, 64, 1000),
    (8, 16, 8, 100), (256, 4096, 256, 65536)])
def test_diagonal_table_range(binding, buckets, max_rel, span, L):
    """The diagonal tables cover every tile offset m whose distances
    [128 m - 127, 128 m + 127] are not all saturated (checked with the oracle's
    index function), with at most one offset of slack on each side."""
    from oracle import rel_index
    lay = binding.df_attn_workspace_layout(3, 4, L, 64, buckets=buckets, max_rel=max_rel, span=span)
    lay128 = binding.df_attn_workspace_layout(3, 4, L, 128, buckets=buckets, max_rel=max_rel, span=span)
    nkb = (L + 127) // 128
    top = 2 * span - 1
    near = []
    for m in range(-(nkb - 1), nkb):
        u = rel_index(np.arange(128 * m - 127, 128 * m + 128), buckets, max_rel, span)
        if not (np.all(u == top) or np.all(u == 0)):
            near.append(m)
    m0, n = lay["diag_m0"], lay["n_diag"]
    assert m0 <= min(near) and m0 + n - 1 >= max(near)
    assert n <= len(near) + 2
    rows = (n + 1) * 128 * 4 * 64 * 2
    assert lay["diag_pq"] - lay["diag_pk"] >= rows and lay["total"] - lay["diag_pq"] >= rows
    # head size 128: the same offsets, rows twice as wide
    assert (lay128["diag_m0"], lay128["n_diag"]) == (m0, n)
    assert lay128["diag_pq"] - lay128["diag_pk"] >= 2 * rows and lay128["total"] - lay128["diag_pq"] >= 2 * rows


def _fwd_raw(binding, **over):
    """Call df_attn_fwd with fake (never dereferenced) aligned pointers."""
    a = dict(q=0x10000, k=0x20000, v=0x30000, pk=0x40000, pq=0x50000, mask=0x60000, cu=None,
             B=2, H=2, L=64, T=128, d=64, buckets=256, max_rel=512, span=256, dtype=0,
             out=0x70000, ws=0x100000, ws_bytes=1 << 30)
    a.update(over)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return binding.raw_library.df_attn_fwd(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["pk"]), vp(a["pq"]), vp(a["mask"]), vp(a["cu"]),
        a["B"], a["H"], a["L"], a["T"], a["d"], a["buckets"], a["max_rel"], a["span"], a["dtype"],
        vp(a["out"]), vp(a["ws"]), a["ws_bytes"], None)


def test_host_side_rejections(binding):
    b = binding
    assert _fwd_raw(b, mask=None) == b.DF_ERR_INVALID_ARG               # neither mask nor cu
    assert _fwd_raw(b, cu=0x80000) == b.DF_ERR_INVALID_ARG              # both
    assert _fwd_raw(b, d=96) == b.DF_ERR_UNSUPPORTED
    assert _fwd_raw(b, T=127) == b.DF_ERR_INVALID_ARG                   # padded needs T = B*L
    assert _fwd_raw(b, mask=None, cu=0x80000, T=129) == b.DF_ERR_INVALID_ARG  # T > B*L
    assert _fwd_raw(b, q=0x10008) == b.DF_ERR_ALIGNMENT
    assert _fwd_raw(b, out=0x70004) == b.DF_ERR_ALIGNMENT
    assert _fwd_raw(b, ws=0x100010) == b.DF_ERR_ALIGNMENT
    assert _fwd_raw(b, ws_bytes=1000) == b.DF_ERR_WORKSPACE
    assert _fwd_raw(b, ws=None) == b.DF_ERR_WORKSPACE
    assert _fwd_raw(b, v=None) == b.DF_ERR_INVALID_ARG
    assert _fwd_raw(b, dtype=5) == b.DF_ERR_INVALID_ARG
    assert _fwd_raw(b, B=-1) == b.DF_ERR_INVALID_ARG
    assert b.raw_library.df_attn_get_device_status(None, None) == b.DF_ERR_INVALID_ARG
    assert b.raw_library.df_rel_index_table(256, 512, 256, 0, ctypes.c_void_p(0x1000),
                                            None) == b.DF_ERR_INVALID_ARG


def test_pack_entry_points_check_arguments_on_the_host(binding):
    lib = binding.raw_library
    ok_ptr, odd_ptr = ctypes.c_void_p(16 * 1024), ctypes.c_void_p(16 * 1024 + 8)
    inv = ctypes.c_void_p(64 * 1024)
    # rows must be 16-byte multiples, pointers 16-byte aligned, sizes positive
    assert lib.df_pack_rows(ok_ptr, inv, inv, 4, 8, ok_ptr, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_pack_rows(ok_ptr, inv, inv, 0, 16, ok_ptr, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_pack_rows(odd_ptr, inv, inv, 4, 16, ok_ptr, None) == binding.DF_ERR_ALIGNMENT
    assert lib.df_pack_rows(None, inv, inv, 4, 16, ok_ptr, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_unpack_rows(ok_ptr, inv, 4, 24, ok_ptr, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_unpack_rows(ok_ptr, inv, 4, 32, odd_ptr, None) == binding.DF_ERR_ALIGNMENT
    assert lib.df_pack_info(ok_ptr, 0, 8, inv, inv, inv, inv, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_pack_info(ok_ptr, 2, 0, inv, inv, inv, inv, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_pack_info(None, 2, 8, inv, inv, inv, inv, None) == binding.DF_ERR_INVALID_ARG


def test_linear_checks_arguments_on_the_host(binding):
    lib = binding.raw_library
    p = ctypes.c_void_p(16 * 1024)
    odd = ctypes.c_void_p(16 * 1024 + 4)
    arr = (ctypes.c_void_p * 3)(16 * 1024, 16 * 1024, 16 * 1024)
    assert lib.df_linear(p, 4, 64, 0, arr, None, 256, arr, 0, binding.DF_BF16, None, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_linear(p, 4, 64, 4, arr, None, 256, arr, 0, binding.DF_BF16, None, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_linear(p, 0, 64, 1, arr, None, 256, arr, 0, binding.DF_BF16, None, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_linear(p, 4, 48, 1, arr, None, 256, arr, 0, binding.DF_BF16, None, None) == binding.DF_ERR_UNSUPPORTED
    assert lib.df_linear(p, 4, 64, 1, arr, None, 200, arr, 0, binding.DF_BF16, None, None) == binding.DF_ERR_UNSUPPORTED
    assert lib.df_linear(p, 4, 64, 1, arr, None, 256, arr, 0, binding.DF_FP32, None, None) == binding.DF_ERR_UNSUPPORTED
    assert lib.df_linear(odd, 4, 64, 1, arr, None, 256, arr, 0, binding.DF_BF16, None, None) == binding.DF_ERR_ALIGNMENT
    assert lib.df_linear(p, 4, 64, 1, arr, None, 256, arr, 2, binding.DF_BF16, None, None) == binding.DF_ERR_INVALID_ARG


def test_layernorm_checks_arguments_on_the_host(binding):
    lib = binding.raw_library
    p, odd = ctypes.c_void_p(16 * 1024), ctypes.c_void_p(16 * 1024 + 2)
    f = ctypes.c_float
    assert lib.df_layernorm(p, None, p, p, 0, 768, f(1e-7), p, binding.DF_BF16, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_layernorm(p, None, p, p, 4, 768, f(0.0), p, binding.DF_BF16, None) == binding.DF_ERR_INVALID_ARG
    assert lib.df_layernorm(p, None, p, p, 4, 700, f(1e-7), p, binding.DF_BF16, None) == binding.DF_ERR_UNSUPPORTED
    assert lib.df_layernorm(p, None, p, p, 4, 1280, f(1e-7), p, binding.DF_BF16, None) == binding.DF_ERR_UNSUPPORTED
    assert lib.df_layernorm(p, None, p, p, 4, 768, f(1e-7), p, binding.DF_FP32, None) == binding.DF_ERR_UNSUPPORTED
    assert lib.df_layernorm(p, odd, p, p, 4, 768, f(1e-7), p, binding.DF_BF16, None) == binding.DF_ERR_ALIGNMENT


def _bwd_raw(binding, **over):
    """Call df_attn_bwd with fake (never dereferenced) aligned pointers."""
    a = dict(q=0x10000, k=0x20000, v=0x30000, pk=0x40000, pq=0x50000, do=0x58000, mask=0x60000,
             cu=None, B=2, H=2, L=64, T=128, d=64, buckets=256, max_rel=512, span=256, dtype=0,
             dq=0x70000, dk=0x78000, dv=0x80000, dpk=0x88000, dpq=0x90000, ws=0x100000,
             ws_bytes=1 << 40)
    a.update(over)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return binding.raw_library.df_attn_bwd(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["pk"]), vp(a["pq"]), vp(a["do"]), vp(a["mask"]),
        vp(a["cu"]), a["B"], a["H"], a["L"], a["T"], a["d"], a["buckets"], a["max_rel"], a["span"],
        a["dtype"], vp(a["dq"]), vp(a["dk"]), vp(a["dv"]), vp(a["dpk"]), vp(a["dpq"]), vp(a["ws"]),
        a["ws_bytes"], None)


def test_backward_checks_arguments_on_the_host(binding):
    b = binding
    fwd = b.df_attn_workspace_size(2, 2, 64, 64)
    bwd = b.df_attn_bwd_workspace_size(2, 2, 64, 64)
    # the bucket sums alone take 2 tables x T x H x 2 span floats
    assert bwd >= fwd + 2 * 128 * 2 * 512 * 4
    # no bucketing: span = max_rel = 512, twice the bucket-sum tables
    assert b.df_attn_bwd_workspace_size(2, 2, 64, 64, buckets=0, max_rel=512) >= fwd + 2 * 128 * 2 * 1024 * 4
    assert b.df_attn_bwd_workspace_size(2, 2, 64, 48) == 0
    assert _bwd_raw(b, d=96) == b.DF_ERR_UNSUPPORTED
    assert _bwd_raw(b, ws_bytes=bwd - 1) == b.DF_ERR_WORKSPACE
    assert _bwd_raw(b, dpk=None) == b.DF_ERR_INVALID_ARG
    assert _bwd_raw(b, do=None) == b.DF_ERR_INVALID_ARG
    assert _bwd_raw(b, dq=None) == b.DF_ERR_INVALID_ARG
    assert _bwd_raw(b, do=0x58004) == b.DF_ERR_ALIGNMENT
    assert _bwd_raw(b, dv=0x80008) == b.DF_ERR_ALIGNMENT
    assert _bwd_raw(b, mask=None) == b.DF_ERR_INVALID_ARG


def test_host_forward_checks_arguments_on_the_host(binding):
    """df_attn_fwd_host reads cu_seqlens on the host and rejects a bad call
    before any CUDA call (fake device pointers are never touched)."""
    b = binding
    lib = b.raw_library
    cu = np.array([0, 5, 12, 12], dtype=np.int32)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    cu_p = cu.ctypes.data_as(ctypes.c_void_p)
    size = b.df_attn_fwd_host_scratch_size(3, 2, 16, 64, b.DF_BF16)
    assert size > b.df_attn_workspace_size(3, 2, 16, 64)
    assert b.df_attn_fwd_host_scratch_size(3, 2, 16, 48, b.DF_BF16) == 0

    def call(cu_ptr=cu_p, mask=None, T=12, L=16, scratch=0x100000, nbytes=size, group=0):
        return lib.df_attn_fwd_host(vp(0x1000), vp(0x2000), vp(0x3000), vp(0x4000), vp(0x5000),
                                    vp(mask), cu_ptr, 3, 2, L, T, 64, 256, 512, 256, 0, vp(0x6000),
                                    group, vp(scratch), nbytes, None)

    assert call(T=13) == b.DF_ERR_INVALID_ARG          # cu_seqlens[B] != total_tokens
    assert call(L=6) == b.DF_ERR_INVALID_ARG           # a length above L
    assert call(mask=0x7000) == b.DF_ERR_INVALID_ARG   # both mask and cu_seqlens
    assert call(nbytes=size - 1) == b.DF_ERR_WORKSPACE
    assert call(scratch=0x100010) == b.DF_ERR_ALIGNMENT
    assert call(group=-1) == b.DF_ERR_INVALID_ARG
    bad = np.array([0, 7, 5, 12], dtype=np.int32)       # decreasing
    assert call(cu_ptr=bad.ctypes.data_as(ctypes.c_void_p)) == b.DF_ERR_INVALID_ARG


def test_head_size_32_workspace_holds_the_widened_copies(binding):
    """bf16 / fp16 at d = 32 run the d = 64 kernels on zero-widened copies: the
    workspace holds the d = 64 layout plus q, k, v, out and PK, PQ at 64 columns."""
    B, H, L = 4, 24, 2048
    d64 = binding.df_attn_workspace_layout(B, H, L, 64)["total"]
    widened = 4 * B * L * H * 64 * 2 + 2 * 512 * H * 64 * 2
    assert binding.df_attn_workspace_size(B, H, L, 32) >= d64 + widened


def _fast_raw(binding, **over):
    """Call df_attn_fwd_fp32_fast with fake (never dereferenced) aligned pointers."""
    a = dict(q=0x10000, k=0x20000, v=0x30000, pk=0x40000, pq=0x50000, mask=0x60000, cu=None,
             B=2, H=2, L=64, T=128, d=64, buckets=256, max_rel=512, span=256,
             out=0x70000, ws=0x100000, ws_bytes=1 << 30)
    a.update(over)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return binding.raw_library.df_attn_fwd_fp32_fast(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["pk"]), vp(a["pq"]), vp(a["mask"]), vp(a["cu"]),
        a["B"], a["H"], a["L"], a["T"], a["d"], a["buckets"], a["max_rel"], a["span"],
        vp(a["out"]), vp(a["ws"]), a["ws_bytes"], None)


def test_fast_fp32_host_side_rejections(binding):
    """Every argument error of the fast fp32 mode is caught before anything is
    enqueued (the pointers are never dereferenced)."""
    b = binding
    need = b.df_attn_fwd_fp32_fast_workspace_size(2, 2, 64, 64, 256, 512, 256)
    assert _fast_raw(b, mask=None) == b.DF_ERR_INVALID_ARG               # neither mask nor cu
    assert _fast_raw(b, cu=0x80000) == b.DF_ERR_INVALID_ARG              # both
    assert _fast_raw(b, d=96) == b.DF_ERR_UNSUPPORTED
    assert _fast_raw(b, T=127) == b.DF_ERR_INVALID_ARG                   # padded needs T = B*L
    assert _fast_raw(b, mask=None, cu=0x80000, T=129) == b.DF_ERR_INVALID_ARG  # T > B*L
    assert _fast_raw(b, q=0x10008) == b.DF_ERR_ALIGNMENT
    assert _fast_raw(b, v=0x30004) == b.DF_ERR_ALIGNMENT
    assert _fast_raw(b, pq=0x50008) == b.DF_ERR_ALIGNMENT
    assert _fast_raw(b, ws=0x100010) == b.DF_ERR_ALIGNMENT
    assert _fast_raw(b, ws_bytes=need - 1) == b.DF_ERR_WORKSPACE
    assert _fast_raw(b, ws=None) == b.DF_ERR_WORKSPACE
    assert _fast_raw(b, v=None) == b.DF_ERR_INVALID_ARG
    assert _fast_raw(b, pk=None) == b.DF_ERR_INVALID_ARG
    assert _fast_raw(b, B=-1) == b.DF_ERR_INVALID_ARG


@pytest.mark.parametrize("B,H,L,d", [(2, 2, 64, 64), (16, 12, 512, 64), (4, 8, 2048, 128), (3, 4, 300, 32)])
def test_fast_fp32_workspace_holds_the_fp16_forward_and_copies(binding, B, H, L, d):
    """The fast mode's workspace is the fp16 forward's workspace plus fp16
    copies of q, k, v, out (B L rows) and of PK, PQ."""
    span = 256
    fast = binding.df_attn_fwd_fp32_fast_workspace_size(B, H, L, d, 256, 512, span)
    base = binding.df_attn_workspace_size(B, H, L, d, 256, 512, span)
    assert fast >= base + 4 * B * L * H * d * 2 + 2 * (2 * span * H * d * 2)
    assert fast % 256 == 0
    assert binding.df_attn_fwd_fp32_fast_workspace_size(B, H, L, 96, 256, 512, span) == 0


def test_layout_is_the_same_whatever_the_call_history(binding):
    """The host keeps the bucket function's saturation points of the last few
    parameter sets; layouts (near-tile offsets, sizes) must not depend on which
    sets were used before or in what order (more sets than are kept, so some
    are computed again)."""
    sets = [(256, 512, 256, 8192), (256, 512, 256, 300), (0, 512, 512, 2048), (64, 128, 64, 1000),
            (8, 16, 8, 100), (256, 4096, 256, 65536), (128, 256, 128, 4096), (32, 64, 32, 700),
            (16, 64, 16, 5000), (256, 1024, 256, 3000), (2, 8, 2, 50), (0, 64, 64, 64)]
    first = {}
    for s in sets:
        first[s] = dict(binding.df_attn_workspace_layout(2, 4, s[3], 64, buckets=s[0], max_rel=s[1], span=s[2]))
    for s in reversed(sets + sets[::3]):
        got = dict(binding.df_attn_workspace_layout(2, 4, s[3], 64, buckets=s[0], max_rel=s[1], span=s[2]))
        assert got == first[s], s


def test_binding_refuses_host_tensors_instead_of_computing_on_the_cpu(binding):
    """There is no CPU path: the Python entry points reject tensors that are
    not on a CUDA device before anything reaches the library."""
    import torch
    T, H, d = 64, 2, 64
    q = torch.zeros(T, H, d, dtype=torch.bfloat16)
    pos = torch.zeros(512, H, d, dtype=torch.bfloat16)
    cu = torch.tensor([0, T], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.df_attn_fwd(q, q, q, pos, pos, cu_seqlens=cu, max_seqlen=T)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.df_attn_fwd_fp32_fast(q.float(), q.float(), q.float(), pos.float(), pos.float(),
                                      cu_seqlens=cu, max_seqlen=T)
    with pytest.raises(ValueError, match="float32"):
        binding.df_attn_fwd_fp32_fast(q, q, q, pos, pos, cu_seqlens=cu, max_seqlen=T)
    with pytest.raises(ValueError, match="exactly one"):
        binding.df_attn_fwd(q, q, q, pos, pos)
