"""Pins of the projection oracle (oracle/linear.py): identity weights return
the input, a hand-computed 2 x 2 case, and the stacked-QKV split equals three
separate projections."""

import numpy as np

from oracle import linear


def test_identity_weight_returns_input_plus_bias():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 4))
    b = np.array([1.0, -2.0, 0.5, 0.0])
    (y,) = linear(x, [np.eye(4)], [b])
    np.testing.assert_array_equal(y, x + b)


def test_hand_example():
    x = np.array([[1.0, 2.0], [3.0, 4.0]])
    w = np.array([[1.0, 0.0], [1.0, 1.0], [0.0, -1.0]])   # [N = 3, K = 2]
    (y,) = linear(x, [w], [np.array([0.0, 10.0, 0.0])])
    assert y.tolist() == [[1.0, 13.0, -2.0], [3.0, 17.0, -4.0]]


def test_stacked_weight_split():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 8))
    w = rng.standard_normal((9, 8))
    parts = linear(x, [w[0:3], w[3:6], w[6:9]])
    (whole,) = linear(x, [w])
    np.testing.assert_allclose(np.concatenate(parts, axis=1), whole, rtol=0, atol=1e-12)
