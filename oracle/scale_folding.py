"""Plain CPU oracle of the zero-cost scale folds (numpy, float64).

TEST INFRASTRUCTURE ONLY.  Only the tests may import this module; the library
never does, and it shares no code with the CUDA path.

What it computes, and where the pages state it:
  * attention temperature matching (ATM): a per-head scalar alpha that
    corrects the spread of the attention logits, folded into the dequant
    scale at inference; output head balancing (OHB): a per-layer scalar beta
    that corrects the gain of the output projection, folded the same way --
    "QuantVLA: Scale-Calibrated Post-Training Quantization for
    Vision-Language-Action Models" summary, section 2 (B: ATM, C: OHB; both
    need no extra computation or buffer at inference);
  * channel scaling combined with block Hadamard transforms and dynamic
    per-token quantization -- FoldQuantVLA abstract.

Readings (the pages give no formula):
  R24 a fold multiplies the per-output-channel weight scale: s_w'[n] =
      float32(s_w[n] * f[n]), f = alpha_h on the channels of head h of the
      projection whose logits it corrects, f = beta on every channel of the
      output projection; the integer GEMM and the codes are unchanged.
  R25 channel scaling: one positive factor c[k] per input channel,
      W' = W diag(c) offline and x' = x diag(1/c) online, both before the
      block rotation, so x' W'^T = x W^T.
"""
from __future__ import annotations

import numpy as np

from oracle.vqlin_oracle import (bf16_to_f64, block_hadamard_rotate, int_gemm, linear_epilogue, rtn_static,
                                 rtn_symmetric_rows)


def fold_output_scales(sw, factor) -> np.ndarray:
    """s_w' = float32(s_w * f) per output channel (R24)."""
    return (np.asarray(sw, np.float64) * np.asarray(factor, np.float64)).astype(np.float32)


def head_factors(alpha, head_dim: int) -> np.ndarray:
    """Per-channel factors of a projection with len(alpha) heads of head_dim channels."""
    return np.repeat(np.asarray(alpha, np.float64), head_dim)


def linear_quantized_scaled(X_bits, W_bits, bits: int, hadamard_block: int, c=None, out_factor=None,
                            bias_bits=None, act_bits=None, static_scale=None):
    """Whole projection with channel scaling c (R25) and an output-scale fold
    (R24): W' = W diag(c) rotated offline and quantized per channel,
    x' = x diag(1/c) rotated online and quantized per token, integer GEMM,
    epilogue with s_w' = s_w * f.  static_scale: one precomputed activation
    scale for every token instead of the per-token scales (the per-step static
    scales of the Omega-QVLA summary, "Scalatura delle Attivazioni DiT per
    Passo"), codes clamped to the symmetric range."""
    W = bf16_to_f64(W_bits)
    X = bf16_to_f64(X_bits)
    if c is not None:
        c = np.asarray(c, np.float64)
        W = W * c[None, :]
        X = X / c[None, :]
    Wt32 = block_hadamard_rotate(W, hadamard_block).astype(np.float32)
    wq, sw = rtn_symmetric_rows(Wt32, bits)
    Xt32 = block_hadamard_rotate(X, hadamard_block).astype(np.float32)
    abits = bits if act_bits is None else act_bits
    if static_scale is None:
        xq, sx = rtn_symmetric_rows(Xt32, abits)
    else:
        s = np.float32(static_scale)
        xq, sx = rtn_static(Xt32, abits, s), np.full(Xt32.shape[0], s, dtype=np.float32)
    if out_factor is not None:
        sw = fold_output_scales(sw, out_factor)
    acc = int_gemm(xq, wq)
    y = linear_epilogue(acc, sx, sw, bias_bits)
    return dict(xq=xq, sx=sx, wq=wq, sw=sw, acc=acc, y=y)
