"""Pins of the composite SVD.Hadamard block-rotation oracle
(oracle/composite_rotation.py) against what the mathematics fixes."""
import os

import numpy as np
import pytest

from oracle import composite_rotation as cr
from oracle import vqlin_oracle as o
from synth import activations, weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_zigzag():
    vals = {}
    for ln in open(os.path.join(GOLDEN, "zigzag_case.txt")):
        if ln.strip() and not ln.startswith("#"):
            k, *v = ln.split()
            vals[k] = [int(x) for x in v]
    return vals


def test_zigzag_golden_case():
    g = _golden_zigzag()
    norms = np.array(g["norms"], dtype=np.float64)
    W = np.diag(norms)                      # column k has norm norms[k]
    assert list(cr.zigzag_permutation(W, 4)) == g["perm"]


@pytest.mark.parametrize("K,b", [(256, 64), (512, 128), (128, 128)])
def test_zigzag_is_a_balanced_permutation(K, b):
    W = o.bf16_to_f64(weights(64, K, spike_frac=0.01, spike_scale=10, seed=1))
    perm = cr.zigzag_permutation(W, b)
    assert sorted(perm) == list(range(K))
    norms = np.sqrt((W * W).sum(0))[perm].reshape(K // b, b)
    # every block takes one channel from each round of K/b consecutive ranks
    ranks = np.argsort(np.argsort(-np.sqrt((W * W).sum(0)), kind="stable"), kind="stable")[perm].reshape(K // b, b)
    for r in range(b):
        assert sorted(ranks[:, r]) == list(range(r * (K // b), (r + 1) * (K // b)))
    assert norms.shape == (K // b, b)


@pytest.mark.parametrize("N,K,b", [(64, 256, 64), (32, 256, 128), (300, 512, 128)])
def test_block_rotations_are_orthogonal_with_fixed_signs(N, K, b):
    W = o.bf16_to_f64(weights(N, K, seed=2))
    perm = cr.zigzag_permutation(W, b)
    R = cr.block_rotations(W, perm, b)
    H = o.sylvester_hadamard(b).astype(np.float64) / np.sqrt(b)
    for Rj in R:
        assert np.abs(Rj @ Rj.T - np.eye(b)).max() < 1e-12
        V = Rj @ H.T                         # R_j H^T = V_j (H orthogonal, symmetric)
        big = np.argmax(np.abs(V), axis=0)
        assert np.all(V[big, np.arange(b)] > 0)


@pytest.mark.parametrize("b", [64, 128])
def test_composite_rotation_preserves_the_gemm(b):
    X = o.bf16_to_f64(activations(8, 256, n_outliers=3, outlier_scale=20, seed=3))
    W = o.bf16_to_f64(weights(48, 256, seed=4))
    perm = cr.zigzag_permutation(W, b)
    R = cr.block_rotations(W, perm, b)
    y = cr.composite_rotate(X, perm, R) @ cr.composite_rotate(W, perm, R).T
    exact = X @ W.T
    assert np.linalg.norm(y - exact) <= 1e-12 * np.linalg.norm(exact)


@pytest.mark.parametrize("N,b", [(96, 64), (300, 128), (40, 64)])
def test_composite_rotation_equalises_weight_column_energy(N, b):
    # W_j V_j = U_j S_j has columns s_i u_i; the normalised Hadamard mixes them
    # with weights +-1/sqrt(b), so every rotated column has squared norm
    # sum_i s_i^2 / b = ||W_j||_F^2 / b
    K = 256
    W = o.bf16_to_f64(weights(N, K, spike_frac=0.01, spike_scale=10, seed=5))
    perm = cr.zigzag_permutation(W, b)
    Wt = cr.composite_rotate(W, perm, cr.block_rotations(W, perm, b))
    for j in range(K // b):
        blk = Wt[:, j * b:(j + 1) * b]
        want = np.linalg.norm(W[:, perm[j * b:(j + 1) * b]]) / np.sqrt(b)
        assert np.allclose(np.linalg.norm(blk, axis=0), want, rtol=1e-12, atol=0)


def test_orthogonal_descending_columns_reduce_to_block_hadamard():
    # columns that are orthogonal and already in descending norm order within
    # each block have V_j = I, so the composite rotation is the block Hadamard
    # of the permuted channels
    K, b = 128, 64
    norms = np.linspace(10.0, 1.0, K)
    W = np.zeros((K, K))
    W[np.arange(K), np.arange(K)] = norms    # column k = norms[k] e_k
    perm = cr.zigzag_permutation(W, b)
    R = cr.block_rotations(W, perm, b)
    for Rj in R:
        assert np.allclose(Rj, o.sylvester_hadamard(b) / np.sqrt(b), atol=1e-13)
    X = o.bf16_to_f64(activations(4, K, seed=6))
    assert np.allclose(cr.composite_rotate(X, perm, R), o.block_hadamard_rotate(X[:, perm], b), atol=1e-12)


@pytest.mark.parametrize("bits,abits", [(4, 4), (8, 8), (4, 8)])
def test_composite_projection_within_rtn_error_bound(bits, abits):
    M, N, K, b = 8, 32, 256, 64
    xb = activations(M, K, n_outliers=4, outlier_scale=20, seed=7)
    wb = weights(N, K, seed=8)
    r = cr.linear_quantized_composite(xb, wb, bits, b, act_bits=abits)
    x, w = o.bf16_to_f64(xb), o.bf16_to_f64(wb)
    exact = x @ w.T
    xt = np.abs(cr.composite_rotate(x, r["perm"], r["R"]))
    wt = np.abs(cr.composite_rotate(w, r["perm"], r["R"]))
    sx = r["sx"].astype(np.float64)[:, None]
    sw = r["sw"].astype(np.float64)[None, :]
    bound = xt.sum(1)[:, None] * sw / 2 + wt.sum(1)[None, :] * sx / 2 + K * sx * sw / 4
    bound = bound * (1 + 1e-5) + np.abs(exact) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(o.bf16_to_f64(r["y"]) - exact) <= bound)
