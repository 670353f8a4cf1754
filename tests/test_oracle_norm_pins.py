"""Pins of the AdaLayerNorm oracle (oracle/norm_fusion.py): a hand-computed
case, the normalisation's invariants, the modulation, and the quantizer's
bounds on its output."""
import numpy as np
import pytest

from oracle import norm_fusion as nf
from oracle import vqlin_oracle as o
from synth import activations, sub_rng


def test_hand_case():
    # x = 1, 2, 3, 4: mean 5/2, population variance 5/4, so x^ = (x - 5/2) / sqrt(5/4)
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    y = nf.ada_layer_norm(x, np.zeros(4), np.zeros(4), 0.0)
    r = np.sqrt(1.25)
    np.testing.assert_allclose(y[0], [-1.5 / r, -0.5 / r, 0.5 / r, 1.5 / r], rtol=0, atol=1e-15)
    # printed to 6 places: -1.341641, -0.447214
    assert abs(y[0, 0] + 1.341641) < 1e-6 and abs(y[0, 1] + 0.447214) < 1e-6
    # eps enters under the root: var + eps = 5/4 + 3/4 = 2
    y2 = nf.ada_layer_norm(x, np.zeros(4), np.zeros(4), 0.75)
    np.testing.assert_allclose(y2[0], (x[0] - 2.5) / np.sqrt(2.0), rtol=0, atol=1e-15)


def test_normalised_rows_have_zero_mean_and_unit_variance():
    X = o.bf16_to_f64(activations(9, 512, n_outliers=5, outlier_scale=30, seed=3))
    y = nf.ada_layer_norm(X, np.zeros(512), np.zeros(512), 0.0)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-13)
    np.testing.assert_allclose((y * y).mean(axis=1), 1.0, rtol=1e-13)


def test_invariant_to_a_per_token_offset_and_positive_scale():
    X = o.bf16_to_f64(activations(5, 256, seed=4))
    z = np.zeros(256)
    base = nf.ada_layer_norm(X, z, z, 0.0)
    shifted = nf.ada_layer_norm(X + np.arange(5)[:, None] * 7.0, z, z, 0.0)
    scaled = nf.ada_layer_norm(X * np.array([0.5, 2.0, 3.0, 10.0, 1e-3])[:, None], z, z, 0.0)
    np.testing.assert_allclose(shifted, base, atol=1e-12)
    np.testing.assert_allclose(scaled, base, atol=1e-12)


def test_modulation():
    X = o.bf16_to_f64(activations(4, 128, seed=5))
    rng = sub_rng(6, "mod")
    scale, shift = rng.normal(0, 0.3, 128), rng.normal(0, 0.5, 128)
    base = nf.ada_layer_norm(X, np.zeros(128), np.zeros(128), 1e-6)
    y = nf.ada_layer_norm(X, scale, shift, 1e-6)
    np.testing.assert_allclose(y, base * (1 + scale)[None, :] + shift[None, :], rtol=0, atol=1e-14)
    # scale = -1 leaves the shift alone, for every token
    only = nf.ada_layer_norm(X, -np.ones(128), shift, 1e-6)
    np.testing.assert_array_equal(only, np.broadcast_to(shift, only.shape))


@pytest.mark.parametrize("bits,hb", [(4, 128), (8, 64), (4, 0)])
def test_quantized_output_bounds(bits, hb):
    Xb = activations(7, 1024, n_outliers=10, outlier_scale=30, seed=7)
    rng = sub_rng(8, "mod", bits, hb)
    scale, shift = rng.normal(0, 0.2, 1024), rng.normal(0, 0.2, 1024)
    q, s = nf.adaln_hadamard_quant(Xb, scale, shift, 1e-6, bits, hb)
    qmax = o.qmax_of(bits)
    assert q.min() >= -qmax and q.max() <= qmax
    v = nf.adaln_rotated_f64(Xb, scale, shift, 1e-6, hb).astype(np.float32).astype(np.float64)
    err = np.abs(v - q.astype(np.float64) * s.astype(np.float64)[:, None])
    assert np.all(err <= s.astype(np.float64)[:, None] * (0.5 + 1e-6))
    # the absmax element of every row reaches +-qmax
    assert np.all(np.abs(q).max(axis=1) == qmax)
