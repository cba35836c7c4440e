"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (max-abs / rel-L2): bf16 3e-2 / 1e-2, fp16 1e-2 / 3e-3, strict fp32
1e-5 max-abs.  Every row is compared on the tiny, v3-base padded and
heavy-padding workloads; seeded (sequence, head, row) samples on the packed
varlen and long-context workloads.
"""

import numpy as np
import pytest
import torch

from exact_attention_deberta_gb300 import synth
from oracle import rel_index

from _parity import TOL, assert_close, errors, gpu_rows, oracle_full, oracle_sampled, run_gpu, \
    sample_triples

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("buckets,max_rel,span,max_len", [
    (256, 512, 256, 8192), (256, 512, 256, 8320), (0, 512, 512, 2048), (8, 16, 8, 100),
    (64, 128, 64, 1000), (256, 4096, 256, 65536)])
def test_index_table_exhaustive(lib, buckets, max_rel, span, max_len):
    got = lib.df_rel_index_table(buckets, max_rel, span, max_len).cpu().numpy()
    r = np.arange(-(max_len - 1), max_len)
    want = rel_index(r, buckets, max_rel, span)
    assert np.array_equal(got, want)


def _read_ws(ws, lay, name, dtype, count):
    off = lay[name]
    nbytes = count * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype).cpu()


@pytest.mark.parametrize("name", ["v3base_padded_bf16", "packed_varlen_h12d64", "v2xl_heavypad_fp16"])
def test_plan_worklist_and_scalars(lib, name):
    x = synth.make_inputs(name)
    dev = {n: None if getattr(x, n) is None else getattr(x, n).cuda()
           for n in ("q", "k", "pk", "pq", "key_mask", "cu_seqlens")}
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    if x.w.layout == "padded":
        out, ws = lib.df_attn_plan(dev["q"], dev["k"], dev["pk"], dev["pq"], key_mask=dev["key_mask"], **kw)
        B, L = x.key_mask.shape
    else:
        out, ws = lib.df_attn_plan(dev["q"], dev["k"], dev["pk"], dev["pq"], cu_seqlens=dev["cu_seqlens"],
                                   max_seqlen=x.w.L, **kw)
        B, L = x.cu_seqlens.numel() - 1, x.w.L
    torch.cuda.synchronize()
    lay = lib.df_attn_workspace_layout(B, x.w.H, L, x.w.d, **kw)
    hdr = _read_ws(ws, lay, "header", torch.int32, 16).numpy()
    assert hdr[0] == 0
    # host recomputation of the longest-first work list
    slices = x.seq_slices()
    nblk = [(n + 127) // 128 for _, n in slices]
    order = sorted(range(len(slices)), key=lambda s: (-nblk[s], s))
    want = [(slices[s][0], slices[s][1], h, b) for s in order for h in range(x.w.H) for b in range(nblk[s])]
    assert hdr[2] == len(want)
    items = _read_ws(ws, lay, "items", torch.int32, 4 * len(want)).numpy().reshape(-1, 4)
    assert [tuple(map(int, it)) for it in items] == want
    # saturation points of the index table
    lt = lay["table_half"]
    r = np.arange(-(lt - 1), lt)
    idx = rel_index(r, x.w.buckets, x.w.max_rel, x.w.span)
    top = 2 * x.w.span - 1
    assert hdr[3] == (r[idx == top].min() if np.any(idx == top) else hdr[3])
    assert hdr[4] == (r[idx == 0].max() if np.any(idx == 0) else hdr[4])
    got_idx = _read_ws(ws, lay, "idx_table", torch.int32, 2 * lt - 1).numpy()
    assert np.array_equal(got_idx, idx)
    # position scalars of far tiles (log2-scaled dot products), checked in float64
    tp = lay["t_pad"]
    scal = _read_ws(ws, lay, "scalars", torch.float32, x.w.H * 4 * tp).numpy().reshape(x.w.H, 4, tp)
    q = x.q.double().reshape(-1, x.w.H, x.w.d).numpy()
    k = x.k.double().reshape(-1, x.w.H, x.w.d).numpy()
    pk, pq = x.pk.double().numpy(), x.pq.double().numpy()
    ks = 1.4426950408889634 / np.sqrt(3.0 * x.w.d)
    valid = (x.key_mask.reshape(-1).numpy() != 0) if x.key_mask is not None else np.ones(q.shape[0], bool)
    T = q.shape[0]
    for h in range(x.w.H):
        want4 = np.stack([q[:, h] @ pk[0, h], q[:, h] @ pk[top, h], k[:, h] @ pq[0, h], k[:, h] @ pq[top, h]]) * ks
        got4 = scal[h, :, :T]
        np.testing.assert_allclose(got4[:, valid], want4[:, valid], rtol=1e-5, atol=1e-4)
        assert np.all(np.isneginf(got4[2:, ~valid]))
    # padded query rows are zeroed by the planner
    if x.key_mask is not None:
        o = out.reshape(-1, x.w.H, x.w.d)[torch.from_numpy(~valid).cuda()]
        assert torch.all(o == 0)


@pytest.mark.parametrize("name", ["v3base_padded_bf16", "packed_varlen_h12d64", "packed_varlen_h6d128"])
def test_plan_diagonal_tables(lib, name):
    """Row r of the diagonal tables is PK / PQ at idx(128 diag_m0 - 127 + r),
    byte for byte, so that diagonal t of tile offset m (row 128 (m - diag_m0)
    + t) is PK / PQ at idx(128 m - 127 + t)."""
    x = synth.make_inputs(name)
    dev = {n: None if getattr(x, n) is None else getattr(x, n).cuda()
           for n in ("q", "k", "pk", "pq", "key_mask", "cu_seqlens")}
    kw = dict(buckets=x.w.buckets, max_rel=x.w.max_rel, span=x.w.span)
    if x.w.layout == "padded":
        _, ws = lib.df_attn_plan(dev["q"], dev["k"], dev["pk"], dev["pq"], key_mask=dev["key_mask"], **kw)
        B, L = x.key_mask.shape
    else:
        _, ws = lib.df_attn_plan(dev["q"], dev["k"], dev["pk"], dev["pq"], cu_seqlens=dev["cu_seqlens"],
                                 max_seqlen=x.w.L, **kw)
        B, L = x.cu_seqlens.numel() - 1, x.w.L
    torch.cuda.synchronize()
    lay = lib.df_attn_workspace_layout(B, x.w.H, L, x.w.d, **kw)
    n, m0 = lay["n_diag"], lay["diag_m0"]
    assert n > 0
    rows = 128 * (n + 1)
    r = 128 * m0 - 127 + np.arange(rows)
    u = torch.from_numpy(rel_index(r, **kw).astype(np.int64))
    for name_t, src in (("diag_pk", x.pk), ("diag_pq", x.pq)):
        got = _read_ws(ws, lay, name_t, torch.int16, rows * x.w.H * x.w.d).view(rows, x.w.H, x.w.d)
        want = src.view(torch.int16)[u]
        assert torch.equal(got, want), name_t
        # diagonal t of offset m, as the near-tile kernels address it
        for m in (m0, m0 + n - 1):
            t = np.arange(256)
            um = torch.from_numpy(rel_index(128 * m - 127 + t, **kw).astype(np.int64))
            assert torch.equal(got[128 * (m - m0) + t], src.view(torch.int16)[um]), (name_t, m)


FULL = ["tiny_fp32", "tiny_fp32_pad97", "v3base_padded_bf16", "v2xl_heavypad_fp16"]


@pytest.mark.parametrize("name", FULL)
def test_parity_all_rows(lib, name):
    x = synth.make_inputs(name)
    out = run_gpu(lib, x)
    ref = oracle_full(x)
    got = out.double().cpu().numpy()
    if x.key_mask is not None:
        live = x.key_mask.numpy() != 0
        assert np.all(got[~live] == 0.0)
    assert_close(got, ref, x.w.dtype, name)


SAMPLED = ["packed_varlen_h12d64", "packed_varlen_h6d128", "long_packed_fp32",
           "long_packed_h12d64", "long_packed_h8d128"]


@pytest.mark.parametrize("name", SAMPLED)
def test_parity_sampled_rows(lib, name):
    x = synth.make_inputs(name)
    out = run_gpu(lib, x)
    triples = sample_triples(x, 384, x.w.seed + 1000)
    ref = oracle_sampled(x, triples)
    keys = sorted(ref)
    got = gpu_rows(x, out, keys)
    want = np.stack([ref[k] for k in keys])
    assert_close(got, want, x.w.dtype, name)
    assert torch.isfinite(out).all()
    assert lib.df_attn_last_launch_count() >= 2


EDGE = [
    ("packed", "bf16", 64, [1, 1, 2, 127, 128, 129, 255, 257, 0, 3]),
    ("packed", "fp16", 128, [640, 1, 700, 0]),
    ("packed", "fp32", 64, [1, 65, 191, 0, 300]),
    ("padded", "bf16", 128, [1, 0, 77, 200]),
    ("padded", "fp16", 64, [512, 0, 1, 333]),
    ("padded", "fp32", 128, [19, 64, 0]),
]


@pytest.mark.parametrize("layout,dtype,d,lengths", EDGE)
def test_edge_lengths(lib, layout, dtype, d, lengths):
    L = max(max(lengths), 1)
    x = synth.custom_inputs(layout=layout, dtype=dtype, H=3, d=d, lengths=lengths, L=L, seed=sum(lengths))
    out = run_gpu(lib, x)
    ref = oracle_full(x)
    assert_close(out.double().cpu().numpy(), ref, dtype, f"{layout}-{dtype}-d{d}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_arbitrary_mask_pattern(lib, dtype):
    """Factorized mask with holes (not right-padded): keys and rows drop out anywhere."""
    x = synth.custom_inputs(layout="padded", dtype=dtype, H=2, d=64, lengths=[300, 300, 300], L=300, seed=4)
    m = x.key_mask.clone()
    g = torch.Generator().manual_seed(0)
    m[0] = (torch.rand(300, generator=g) < 0.7).to(torch.uint8)
    m[1, 100:230] = 0
    m[2, :] = 0
    m[2, 299] = 1
    x.key_mask = m
    out = run_gpu(lib, x)
    ref = oracle_full(x)
    assert_close(out.double().cpu().numpy(), ref, dtype, "holes")


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("fp16", 64), ("bf16", 128)])
def test_mask_holes_in_far_tiles(lib, dtype, d):
    """Long padded rows (far tiles exist: 13 key blocks) with key-mask holes in
    both near and far tiles, a row whose valid keys are all far from it, and a
    ragged last key block; checked on every row."""
    L = 1600
    x = synth.custom_inputs(layout="padded", dtype=dtype, H=2, d=d, lengths=[L, L, 1500], L=L, seed=17)
    m = x.key_mask.clone()
    g = torch.Generator().manual_seed(3)
    m[0] = (torch.rand(L, generator=g) < 0.6).to(torch.uint8)
    m[1] = 0
    m[1, 1200:1210] = 1          # rows 0..700 see only far keys
    m[1, 1599] = 1
    m[2, 1400:1500] = 0          # a hole at the end of a ragged sequence
    m[2, 0:40] = 0
    x.key_mask = m
    out = run_gpu(lib, x)
    ref = oracle_full(x)
    assert_close(out.double().cpu().numpy(), ref, dtype, f"far-holes-{dtype}-d{d}")


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("fp16", 64), ("bf16", 128), ("fp16", 128)])
@pytest.mark.parametrize("buckets,max_rel,span", [(0, 300, 300), (32, 64, 32), (256, 512, 128), (16, 4096, 16)])
def test_other_position_parameters(lib, buckets, max_rel, span, dtype, d):
    x = synth.custom_inputs(layout="packed", dtype=dtype, H=2, d=d, lengths=[900, 64, 1500], L=1500,
                            seed=buckets + max_rel + d, buckets=buckets, max_rel=max_rel, span=span)
    out = run_gpu(lib, x)
    triples = sample_triples(x, 200, 7)
    ref = oracle_sampled(x, triples)
    keys = sorted(ref)
    assert_close(gpu_rows(x, out, keys), np.stack([ref[k] for k in keys]), dtype,
                 f"params-{dtype}-d{d}")


@pytest.mark.parametrize("scale", [4.0, 16.0])
@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("fp16", 64), ("bf16", 128), ("fp16", 128)])
def test_large_logits(lib, dtype, d, scale):
    """Q, K, PK and PQ drawn from N(0, scale^2) (V from N(0, 1)): logits reach
    thousands of raw score units, so the position terms must keep their
    precision on near tiles as well as far ones.  Every row of a packed batch
    whose longest sequence has near and far tiles."""
    x = synth.custom_inputs(layout="packed", dtype=dtype, H=2, d=d, lengths=[1800, 700, 129], L=1800,
                            seed=int(scale) + d, scale=scale)
    out = run_gpu(lib, x)
    assert_close(out.double().cpu().numpy(), oracle_full(x), dtype, f"scale{scale:g}-{dtype}-d{d}")


@pytest.mark.parametrize("d", [64, 128])
def test_beyond_8192_tokens(lib, d):
    """A 16384-token sequence (and a short one) in packed mode: sampled rows,
    tile edges included, against the oracle."""
    x = synth.custom_inputs(layout="packed", dtype="bf16", H=2, d=d, lengths=[16384, 300], L=16384,
                            seed=40 + d)
    out = run_gpu(lib, x)
    triples = sample_triples(x, 96, 11)
    triples += [(0, 1, 8191), (0, 0, 8192), (0, 1, 16383), (0, 0, 16256)]
    ref = oracle_sampled(x, triples)
    keys = sorted(ref)
    assert_close(gpu_rows(x, out, keys), np.stack([ref[k] for k in keys]), "bf16", f"L16384-d{d}")


def test_packed_matches_padded(lib):
    lens = [300, 17, 129, 513]
    xp = synth.custom_inputs(layout="packed", dtype="bf16", H=4, d=64, lengths=lens, L=513, seed=21)
    L = 513
    cu = xp.cu_seqlens.numpy()
    pad = lambda t: torch.stack([torch.nn.functional.pad(t[cu[s]:cu[s + 1]], (0, 0, 0, 0, 0, L - lens[s]))
                                 for s in range(len(lens))])  # noqa: E731
    mask = torch.zeros(len(lens), L, dtype=torch.uint8)
    for s, n in enumerate(lens):
        mask[s, :n] = 1
    kw = dict(buckets=256, max_rel=512, span=256)
    op = lib.df_attn_fwd(xp.q.cuda(), xp.k.cuda(), xp.v.cuda(), xp.pk.cuda(), xp.pq.cuda(),
                         cu_seqlens=xp.cu_seqlens.cuda(), max_seqlen=L, **kw)
    od = lib.df_attn_fwd(pad(xp.q).cuda(), pad(xp.k).cuda(), pad(xp.v).cuda(), xp.pk.cuda(), xp.pq.cuda(),
                         key_mask=mask.cuda(), **kw)
    torch.cuda.synchronize()
    for s, n in enumerate(lens):
        a = op[cu[s]:cu[s + 1]].float()
        b = od[s, :n].float()
        assert torch.max(torch.abs(a - b)).item() <= 1e-2


def test_masked_rows_do_not_leak(lib):
    x = synth.make_inputs("v3base_padded_bf16")
    base = run_gpu(lib, x).clone()
    dead = x.key_mask == 0
    for t in (x.q, x.k, x.v):
        noise = torch.randn(t[dead].shape, generator=torch.Generator().manual_seed(1)) * 100
        t[dead] = noise.to(t.dtype)
    again = run_gpu(lib, x)
    assert torch.equal(base, again)


def test_unreachable_position_rows_do_not_matter(lib):
    x = synth.custom_inputs(layout="packed", dtype="fp16", H=2, d=64, lengths=[128, 100], L=128, seed=3)
    base = run_gpu(lib, x).clone()
    reach = np.unique(rel_index(np.arange(-127, 128), 256, 512, 256))
    other = torch.from_numpy(np.setdiff1d(np.arange(512), reach))
    x.pk[other] = 30.0
    x.pq[other] = -30.0
    assert torch.equal(base, run_gpu(lib, x))


def test_zero_sequences_and_status(lib):
    x = synth.custom_inputs(layout="packed", dtype="bf16", H=2, d=64, lengths=[0, 0], L=8, seed=1)
    ws = torch.empty(lib.df_attn_workspace_size(2, 2, 8, 64), dtype=torch.uint8, device="cuda")
    out = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    lib.df_attn_fwd(q, q, q, x.pk.cuda(), x.pq.cuda(), cu_seqlens=x.cu_seqlens.cuda(), max_seqlen=8,
                    out=out, workspace=ws)
    assert lib.df_attn_get_device_status(ws) == lib.DF_OK


def test_bad_cu_seqlens_reported_on_device(lib):
    x = synth.custom_inputs(layout="packed", dtype="bf16", H=2, d=64, lengths=[50, 60], L=64, seed=2)
    cu = torch.tensor([0, 50, 300], dtype=torch.int32)   # last length 250 > max_seqlen 64
    ws = torch.empty(lib.df_attn_workspace_size(2, 2, 64, 64), dtype=torch.uint8, device="cuda")
    lib.df_attn_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), x.pk.cuda(), x.pq.cuda(), cu_seqlens=cu.cuda(),
                    max_seqlen=64, workspace=ws)
    assert lib.df_attn_get_device_status(ws) == lib.DF_ERR_INVALID_ARG
    assert lib.df_attn_get_device_status(ws) == lib.DF_OK   # cleared by the read


def test_deterministic(lib):
    x = synth.make_inputs("packed_varlen_h6d128")
    a = run_gpu(lib, x).clone()
    b = run_gpu(lib, x)
    assert torch.equal(a, b)


@pytest.mark.parametrize("layout,dtype,lengths", [("packed", "bf16", [700, 1, 129, 0, 300]),
                                                  ("padded", "fp16", [512, 77, 0, 200]),
                                                  ("packed", "fp32", [333, 64, 1000])])
def test_head_size_32(lib, layout, dtype, lengths):
    """d = 32 (bf16 / fp16: the d = 64 tensor-core kernels on zero-widened heads;
    fp32: the CUDA-core kernel): every row against the oracle, with ragged, empty
    and single-token sequences and far tiles (L up to 1000)."""
    L = max(lengths)
    x = synth.custom_inputs(layout=layout, dtype=dtype, H=4, d=32, lengths=lengths, L=L, seed=len(lengths) + L)
    out = run_gpu(lib, x)
    assert_close(out.double().cpu().numpy(), oracle_full(x), dtype, f"d32-{layout}-{dtype}")
