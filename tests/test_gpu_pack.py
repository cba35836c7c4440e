"""GPU parity of the padded <-> packed conversion against the oracle: the
metadata (cu_seqlens, row list, inverse, T, longest sequence) and the moved
bytes are compared exactly."""

import numpy as np
import pytest
import torch

from oracle import pack_info, pack_rows, unpack_rows

pytestmark = pytest.mark.gpu


def _masks():
    rng = np.random.default_rng(11)
    yield "right_padded", (np.arange(512)[None, :] < rng.integers(0, 513, 16)[:, None]).astype(np.uint8)
    yield "holes", (rng.random((5, 1000)) < 0.3).astype(np.uint8)
    m = (rng.random((6, 1030)) < 0.9).astype(np.uint8)
    m[2] = 0
    m[4] = 1
    yield "empty_and_full_rows", m
    yield "one_long_row", (rng.random((1, 8192)) < 0.7).astype(np.uint8)
    yield "all_empty", np.zeros((3, 77), np.uint8)
    yield "many_rows", (np.arange(96)[None, :] < rng.integers(0, 97, 3000)[:, None]).astype(np.uint8)


MASKS = list(_masks())


@pytest.mark.parametrize("name,mask", MASKS, ids=[n for n, _ in MASKS])
def test_pack_info_matches_oracle(lib, name, mask):
    info = lib.df_pack_info(torch.from_numpy(mask).cuda())
    cu, idx, inv, T, mx = pack_info(mask)
    assert (info.total, info.max_seqlen) == (T, mx)
    assert info.cu_seqlens.cpu().numpy().tolist() == cu.tolist()
    assert info.indices.cpu().numpy().tolist() == idx.tolist()
    assert info.inverse.cpu().numpy().tolist() == inv.tolist()


@pytest.mark.parametrize("name,mask", MASKS, ids=[n for n, _ in MASKS])
@pytest.mark.parametrize("dtype,feat", [(torch.bfloat16, 768), (torch.float16, (24, 64)), (torch.float32, 4),
                                        (torch.uint8, 16)])
def test_pack_and_unpack_move_exact_bytes(lib, name, mask, dtype, feat):
    B, L = mask.shape
    feat = feat if isinstance(feat, tuple) else (feat,)
    g = torch.Generator().manual_seed(B * L)
    x = (torch.randn((B, L) + feat, generator=g) * 7).to(dtype) if dtype != torch.uint8 else \
        torch.randint(0, 256, (B, L) + feat, generator=g, dtype=torch.uint8)
    tokens, cu, info = lib.pack_padded_with_info(x.cuda(), torch.from_numpy(mask).cuda())
    cu_o, idx, inv, T, mx = pack_info(mask)
    row = x[0, 0].numel() * x.element_size()
    xb = x.view(torch.uint8).numpy().reshape(B * L, row)
    want = pack_rows(xb, idx)
    got = tokens.cpu().view(torch.uint8).numpy().reshape(T, row)
    assert np.array_equal(got, want)
    out, valid = lib.unpack_packed(tokens, cu, L, info)
    want_out = unpack_rows(want, inv)
    assert np.array_equal(out.cpu().view(torch.uint8).numpy().reshape(B * L, row), want_out)
    assert np.array_equal(valid.cpu().numpy(), mask != 0)
