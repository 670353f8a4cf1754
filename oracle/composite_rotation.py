"""Plain CPU oracle of the composite SVD.Hadamard block rotation (numpy, float64).

TEST INFRASTRUCTURE ONLY.  Only the tests may import this module; the library
never does, and it shares no code with the CUDA path.

What it computes, and where the pages state it (Omega-QVLA technical summary,
"Rotazione Composita SVD.Hadamard"):
  * "Rotazione SVD": a rotation taken from the singular value decomposition of
    the weight matrix, which makes each weight direction's energy the one its
    singular value fixes;
  * "Rotazione Hadamard": that rotation composed with a normalised Hadamard
    matrix, R = R_SVD . H, which spreads any dominant channel evenly over all
    channels;
  * "Implementazione a Blocchi": instead of one dense C_in x C_in rotation,
    blocks of b channels, after a zig-zag permutation by weight column norm so
    that high- and low-norm channels are spread evenly over the blocks.

Readings (the pages fix no orientation, sign, ordering or dealing rule):
  R20 orientation: the projection is y = x . W^T with W [N, K] (rows = output
      channels).  The rotation acts on the K input channels; the summary's
      R_SVD = U is the left factor of the weight written input-channel-major
      (W^T = U S V^T), i.e. the right singular vectors of W [N, K].
  R21 signs and order: singular values in descending order (numpy's SVD);
      each singular vector's sign chosen so that its largest-magnitude entry
      (the first such entry on ties) is positive.
  R22 blocks: block j holds b consecutive channels of the permuted order; its
      rotation is R_j = V_j . H_b / sqrt(b), V_j from the SVD of W's columns
      of that block (complete, so V_j is b x b even when N < b).  Activations
      are rotated online, x~ = x[:, P] . blockdiag(R_j), weights offline,
      W~ = W[:, P] . blockdiag(R_j), so that x~ . W~^T = x . W^T.
  R23 zig-zag: channels sorted by descending L2 norm of W's column (stable:
      ties keep channel order), then dealt to the K/b blocks in boustrophedon
      rounds: round r gives sorted[r nb + i] to block i for even r and to
      block nb - 1 - i for odd r (nb = K/b); inside a block, channels keep
      their round order.
"""
from __future__ import annotations

import numpy as np

from oracle.vqlin_oracle import bf16_to_f64, int_gemm, linear_epilogue, rtn_symmetric_rows, sylvester_hadamard


def zigzag_permutation(W, b: int) -> np.ndarray:
    """perm[p] = the original channel at position p of the permuted order (R23)."""
    W = np.asarray(W, dtype=np.float64)
    K = W.shape[1]
    if b <= 0 or K % b:
        raise ValueError("K must be a positive multiple of the block")
    nb = K // b
    norms = np.sqrt((W * W).sum(axis=0))
    order = np.argsort(-norms, kind="stable")            # descending, ties by channel
    perm = np.empty(K, dtype=np.int64)
    for r in range(b):
        for i in range(nb):
            blk = i if r % 2 == 0 else nb - 1 - i
            perm[blk * b + r] = order[r * nb + i]
    return perm


def _sign_fixed(V) -> np.ndarray:
    """Columns of V with their largest-magnitude entry made positive (R21)."""
    V = V.copy()
    for c in range(V.shape[1]):
        k = int(np.argmax(np.abs(V[:, c])))
        if V[k, c] < 0:
            V[:, c] = -V[:, c]
    return V


def block_rotations(W, perm, b: int) -> np.ndarray:
    """R [K/b, b, b]: R_j = V_j . H_b / sqrt(b) per block of the permuted channels (R20-R22)."""
    W = np.asarray(W, dtype=np.float64)
    K = W.shape[1]
    H = sylvester_hadamard(b).astype(np.float64) / np.sqrt(np.float64(b))
    R = np.empty((K // b, b, b), dtype=np.float64)
    for j in range(K // b):
        Wj = W[:, perm[j * b:(j + 1) * b]]
        _, _, Vt = np.linalg.svd(Wj, full_matrices=True)  # Wj = U S Vt, Vt [b, b]
        R[j] = _sign_fixed(Vt.T) @ H
    return R


def composite_rotate(V, perm, R) -> np.ndarray:
    """V[:, perm] . blockdiag(R_j) over the last axis, in float64."""
    V = np.asarray(V, dtype=np.float64)[:, perm]
    nb, b, _ = R.shape
    out = np.einsum("mjk,jkl->mjl", V.reshape(V.shape[0], nb, b), R)
    return out.reshape(V.shape[0], nb * b)


def linear_quantized_composite(X_bits, W_bits, bits: int, b: int, bias_bits=None, act_bits=None):
    """Whole projection with the composite rotation: weights rotated offline
    and quantized per output channel (RTN), activations rotated online and
    quantized per token, exact integer GEMM, float64 epilogue, bf16 output."""
    W = bf16_to_f64(W_bits)
    X = bf16_to_f64(X_bits)
    perm = zigzag_permutation(W, b)
    R = block_rotations(W, perm, b)
    Wt32 = composite_rotate(W, perm, R).astype(np.float32)
    wq, sw = rtn_symmetric_rows(Wt32, bits)
    Xt32 = composite_rotate(X, perm, R).astype(np.float32)
    xq, sx = rtn_symmetric_rows(Xt32, bits if act_bits is None else act_bits)
    acc = int_gemm(xq, wq)
    y = linear_epilogue(acc, sx, sw, bias_bits)
    return dict(perm=perm, R=R, xq=xq, sx=sx, wq=wq, sw=sw, acc=acc, y=y)
