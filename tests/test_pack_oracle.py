"""Pins of the packing oracle (oracle/pack.py) against facts that do not come
from it: a worked example by hand, the closed form for right padding (the
README's case: sequence b owns rows b L .. b L + n_b - 1), the round trip, and
the empty mask."""

import numpy as np

from oracle import pack_info, pack_rows, unpack_rows


def test_worked_example():
    mask = np.array([[1, 1, 0], [1, 0, 1]], dtype=np.uint8)
    cu, idx, inv, T, mx = pack_info(mask)
    assert cu.tolist() == [0, 2, 4]
    assert idx.tolist() == [0, 1, 3, 5]
    assert inv.tolist() == [0, 1, -1, 2, -1, 3]
    assert (T, mx) == (4, 2)


def test_right_padding_closed_form():
    rng = np.random.default_rng(5)
    B, L = 7, 50
    lengths = rng.integers(0, L + 1, size=B)
    mask = (np.arange(L)[None, :] < lengths[:, None]).astype(np.uint8)
    cu, idx, inv, T, mx = pack_info(mask)
    assert cu.tolist() == [0] + np.cumsum(lengths).tolist()
    want = np.concatenate([b * L + np.arange(n) for b, n in enumerate(lengths)])
    assert idx.tolist() == want.tolist()
    assert T == lengths.sum() and mx == lengths.max()
    for b, n in enumerate(lengths):
        assert inv[b * L: b * L + n].tolist() == list(range(cu[b], cu[b] + n))
        assert (inv[b * L + n: (b + 1) * L] == -1).all()


def test_round_trip_restores_valid_rows_and_zeroes_padding():
    rng = np.random.default_rng(6)
    B, L, D = 5, 33, 24
    mask = (rng.random((B, L)) < 0.6).astype(np.uint8)
    x = rng.standard_normal((B, L, D)).astype(np.float32)
    cu, idx, inv, T, mx = pack_info(mask)
    tokens = pack_rows(x, idx)
    assert tokens.shape == (T, D)
    back = unpack_rows(tokens, inv).reshape(B, L, D)
    np.testing.assert_array_equal(back, x * mask[..., None])


def test_empty_mask():
    mask = np.zeros((3, 4), dtype=np.uint8)
    cu, idx, inv, T, mx = pack_info(mask)
    assert cu.tolist() == [0, 0, 0, 0] and idx.size == 0 and (inv == -1).all()
    assert (T, mx) == (0, 0)
    out = unpack_rows(np.zeros((0, 2), np.float32), inv)
    assert out.shape == (12, 2) and not out.any()
