"""Plain CPU oracle of the normalisation fused in front of the projection (numpy, float64).

TEST INFRASTRUCTURE ONLY.  Only the tests may import this module; the library
never does, and it shares no code with the CUDA path.

What it computes, and where the pages state it: the Omega-QVLA technical
summary, "Scalatura delle Attivazioni DiT per Passo" ("Deriva dell'Intervallo
Dinamico"), names the projections whose activation ranges drift over the
denoising steps: the QKV projections that follow an AdaLayerNorm, i.e. whose
input is the time-conditioned normalisation of the residual stream.  The
step before the quantized projection is therefore that normalisation, and
fusing it into the activation kernel saves one write and one read of the
activations.

Readings (the summary gives no formula):
  R28 AdaLayerNorm is the adaptive layer normalisation of diffusion
      transformers: per token, the layer normalisation over the K channels
      without a learned affine part, x^ = (x - mean) / sqrt(var + eps) (var the
      population variance), then the conditioning's per-channel modulation
      y = x^ * (1 + scale[k]) + shift[k]; one (scale, shift) pair of K-vectors
      for all tokens of a call (one conditioning per denoising step).
  R29 fused: the normalised, modulated activation is not rounded to bf16 -- it
      stays in float (float32 on the GPU, float64 here) through the block
      rotation, and is rounded to float32 once before the quantizer decides,
      as for the unfused path (R15).
"""
from __future__ import annotations

import numpy as np

from oracle.vqlin_oracle import bf16_to_f64, block_hadamard_rotate, rtn_static, rtn_symmetric_rows


def ada_layer_norm(X, scale, shift, eps: float) -> np.ndarray:
    """y = (x - mean) / sqrt(var + eps) * (1 + scale) + shift per token, float64 (R28)."""
    X = np.asarray(X, dtype=np.float64)
    mean = X.mean(axis=1, keepdims=True)
    var = ((X - mean) ** 2).mean(axis=1, keepdims=True)
    xhat = (X - mean) / np.sqrt(var + np.float64(eps))
    return xhat * (1.0 + np.asarray(scale, np.float64)[None, :]) + np.asarray(shift, np.float64)[None, :]


def adaln_hadamard_quant(X_bits, scale, shift, eps: float, bits: int, hadamard_block: int, static_scale=None):
    """AdaLayerNorm, block rotation and per-token quantization of bf16 X (R28,
    R29): returns (codes int8 [M, K], scales float32 [M])."""
    Y = ada_layer_norm(bf16_to_f64(X_bits), scale, shift, eps)
    Yt32 = block_hadamard_rotate(Y, hadamard_block).astype(np.float32)
    if static_scale is not None:
        s = np.float32(static_scale)
        return rtn_static(Yt32, bits, s), np.full(Yt32.shape[0], s, dtype=np.float32)
    return rtn_symmetric_rows(Yt32, bits)


def adaln_rotated_f64(X_bits, scale, shift, eps: float, hadamard_block: int) -> np.ndarray:
    """The exact rotated, normalised activations (for locating rounding ties)."""
    return block_hadamard_rotate(ada_layer_norm(bf16_to_f64(X_bits), scale, shift, eps), hadamard_block)

