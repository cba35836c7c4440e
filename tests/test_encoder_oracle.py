"""Pins of the encoder oracle's parts (oracle/encoder.py) against closed forms:
LayerNorm gives zero mean and unit variance rows and a hand-computed case;
GELU at 0, +-1 (x times the standard normal CDF) and far out; a layer whose
weights and biases are all zero reduces to LayerNorm of its input (no
attention contribution, GELU(0) = 0)."""

import math

import numpy as np

from oracle import encoder_layer, gelu, layer_norm


def test_layer_norm_rows_are_standardised():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((6, 256)) * 3 + 1
    y = layer_norm(x, np.ones(256), np.zeros(256), 0.0)
    np.testing.assert_allclose(y.mean(axis=1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=1), 1, atol=1e-10)


def test_layer_norm_hand_case():
    y = layer_norm(np.array([[1.0, 2.0, 3.0]]), np.array([2.0, 2.0, 2.0]), np.array([0.0, 1.0, 0.0]), 1e-7)
    s = math.sqrt(2.0 / 3.0 + 1e-7)
    np.testing.assert_allclose(y, [[-2.0 / s, 1.0, 2.0 / s]], rtol=1e-12)


def test_gelu_values():
    phi1 = 0.5 * (1 + math.erf(1 / math.sqrt(2)))
    np.testing.assert_allclose(gelu(np.array([0.0, 1.0, -1.0, 30.0, -30.0])),
                               [0.0, phi1, -(1 - phi1), 30.0, 0.0], rtol=1e-12, atol=1e-12)


def test_zero_weight_layer_is_layer_norm_of_input():
    hid, H, T = 256, 4, 40
    rng = np.random.default_rng(1)
    h = rng.standard_normal((T, hid))
    z = np.zeros
    p = dict(w_qkv=z((3 * hid, hid)), b_qkv=z(3 * hid), w_o=z((hid, hid)), b_o=z(hid), ln1_g=np.ones(hid),
             ln1_b=z(hid), w_1=z((4 * hid, hid)), b_1=z(4 * hid), w_2=z((hid, 4 * hid)), b_2=z(hid),
             ln2_g=np.ones(hid), ln2_b=z(hid))
    rel = rng.standard_normal((512, hid))
    out = encoder_layer(h, p, rel, np.array([0, 25, 40]), H, buckets=256, max_rel=512, span=256, eps=1e-7)
    np.testing.assert_allclose(out, layer_norm(h, np.ones(hid), z(hid), 1e-7), atol=1e-6)
