"""Pins of the scale-folding oracle (oracle/scale_folding.py): attention
temperature matching / output head balancing folded into the weight scales,
and channel scaling folded into weights and activations."""
import numpy as np
import pytest

from oracle import scale_folding as sf
from oracle import vqlin_oracle as o
from synth import activations, weights


@pytest.mark.parametrize("k", [-3, -1, 1, 2])
def test_power_of_two_fold_scales_the_output_exactly(k):
    # a power-of-two factor is exact in float32 and commutes with bf16 rounding
    M, N, K = 8, 64, 256
    xb, wb = activations(M, K, seed=1), weights(N, K, seed=2)
    plain = sf.linear_quantized_scaled(xb, wb, 4, 128)
    folded = sf.linear_quantized_scaled(xb, wb, 4, 128, out_factor=np.full(N, 2.0 ** k))
    assert np.array_equal(folded["acc"], plain["acc"]) and np.array_equal(folded["xq"], plain["xq"])
    assert np.array_equal(o.bf16_to_f64(folded["y"]), 2.0 ** k * o.bf16_to_f64(plain["y"]))


def test_head_fold_touches_only_its_head():
    M, N, K, hd = 4, 64, 256, 16
    xb, wb = activations(M, K, seed=3), weights(N, K, seed=4)
    alpha = np.array([1.0, 1.25, 1.0, 0.8])
    f = sf.head_factors(alpha, hd)
    assert f.shape == (N,) and np.all(f[16:32] == 1.25) and np.all(f[:16] == 1.0)
    plain = sf.linear_quantized_scaled(xb, wb, 4, 64)
    folded = sf.linear_quantized_scaled(xb, wb, 4, 64, out_factor=f)
    same = f == 1.0
    assert np.array_equal(folded["y"][:, same], plain["y"][:, same])
    # the folded heads are the rounded product of the unrounded output and alpha
    y = plain["acc"] * plain["sx"].astype(np.float64)[:, None] * sf.fold_output_scales(plain["sw"], f)[None, :]
    assert np.array_equal(folded["y"], o.bf16_round(y))


def test_channel_scaling_preserves_the_float_gemm():
    M, N, K = 6, 32, 256
    X, W = o.bf16_to_f64(activations(M, K, seed=5)), o.bf16_to_f64(weights(N, K, seed=6))
    c = np.exp(np.random.default_rng(7).normal(0, 1, K))
    assert np.linalg.norm((X / c) @ (W * c).T - X @ W.T) <= 1e-13 * np.linalg.norm(X @ W.T)


def test_channel_scaling_with_unit_factors_is_the_plain_projection():
    M, N, K = 8, 48, 256
    xb, wb = activations(M, K, n_outliers=3, outlier_scale=20, seed=8), weights(N, K, seed=9)
    a = sf.linear_quantized_scaled(xb, wb, 4, 128, c=np.ones(K))
    b = o.linear_quantized(xb, wb, 4, 128)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["acc"], b["acc"])


def test_channel_scaling_with_a_static_scale():
    # unit factors: the static-scale projection of the main oracle; and a
    # static scale equal to every token's own dynamic scale gives the dynamic
    # projection's codes
    M, N, K = 8, 48, 256
    xb, wb = activations(M, K, n_outliers=3, outlier_scale=20, seed=12), weights(N, K, seed=13)
    s = o.calibrate_static_scale([xb], 4, 128)
    a = sf.linear_quantized_scaled(xb, wb, 4, 128, c=np.ones(K), static_scale=s)
    b = o.linear_quantized(xb, wb, 4, 128, static_scale=s)
    assert np.array_equal(a["xq"], b["xq"]) and np.array_equal(a["y"], b["y"])
    assert np.all(a["sx"] == np.float32(s))
    c = np.exp(np.random.default_rng(14).normal(0, 0.3, K))
    dyn = sf.linear_quantized_scaled(xb[:1], wb, 4, 128, c=c)
    st = sf.linear_quantized_scaled(xb[:1], wb, 4, 128, c=c, static_scale=dyn["sx"][0])
    assert np.array_equal(dyn["xq"], st["xq"]) and np.array_equal(dyn["y"], st["y"])


def test_channel_scaling_moves_outlier_energy_into_the_weights():
    # dividing the outlier channels of x by c and multiplying W's columns by c
    # lowers the activation scale and raises the weight scales, the trade the
    # method makes before the rotation
    M, N, K = 16, 64, 256
    xb = activations(M, K, n_outliers=4, outlier_scale=30, seed=10)
    wb = weights(N, K, seed=11)
    X = o.bf16_to_f64(xb)
    amax = np.abs(X).max(0)
    c = np.sqrt(amax / np.abs(o.bf16_to_f64(wb)).max(0))     # a SmoothQuant-style balance
    plain = sf.linear_quantized_scaled(xb, wb, 4, 0)
    scaled = sf.linear_quantized_scaled(xb, wb, 4, 0, c=c)
    assert scaled["sx"].mean() < plain["sx"].mean() and scaled["sw"].mean() > plain["sw"].mean()
