"""Plain CPU oracle of the quantized linear projection (numpy, float64).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this module; the library never does,
and it shares no code with the CUDA path.

What it computes, and where the pages state it:

  * Block Hadamard rotation with a normalised Hadamard matrix H (H.H^T = I),
    applied block-wise over channels: Omega-QVLA summary, "Rotazione
    Composita SVD.Hadamard" (normalised H; block-wise implementation) and the
    FoldQuantVLA abstract ("block Hadamard transforms").  H is Sylvester's
    construction scaled by 1/sqrt(b); the rotation x~ = x.blockdiag(H_b) is
    applied online to activations and folded offline into the weights, so
    x~.W~^T = x.W^T.
  * Round-to-nearest (RTN) weight quantization: LoopQ abstract ("plain RTN
    matches the calibrated methods").  Symmetric per-output-channel int4 /
    int8, or asymmetric group-wise int4 with a bf16 scale and zero point.
  * Dynamic per-token activation quantization: FoldQuantVLA abstract
    ("dynamic per-token quantization"); the static per-step alternative is
    the Omega-QVLA per-step DiT activation scaling ("Calibrazione per Passo").
  * Native integer execution of W4A4 / W8A8 projections: FoldQuantVLA
    abstract; the int32 accumulator is dequantised by the per-token and
    per-channel scales.
  * Weight-only int4 for the memory-bound action expert: LoopQ abstract
    (the expert is memory-bound, 63% of GPU time).

The pages fix no rounding mode, scale formula, group size or bit packing.
The readings taken here (each a plain textbook choice):
  R1 Sylvester H_b, scaled 1/sqrt(b), b in {64, 128}; blocks are consecutive
     channel ranges [j*b, (j+1)*b).
  R3 symmetric scale = absmax / qmax (qmax = 7 or 127), codes clamped to
     the symmetric range [-qmax, qmax] (absmax scaling never leaves it; a
     static scale can, and then clamps to +-qmax).
  R4 round half to even everywhere; x / s is an IEEE float32 division; the
     decision that produces a code is taken in float32 (the kernel's
     precision) from the float32 rounding of the exact rotated value.
  R5 an all-zero row gives scale 0 and codes 0; an all-zero group gives
     scale 1 and zero point 0.
  R6 asymmetric range forced to include 0; scale rounded up to bf16 so that
     15*s covers the range; zero point rint(-lo/s) stored in bf16.
  R7 per-channel and per-token scales are float32.
  R13 final outputs are rounded once to bf16, round half to even.

Packing (a format of this library; the pages fix none): symmetric codes are
sign-magnitude -- an int4 weight code c is the nibble (c < 0) << 3 | |c|, two
per byte with the even channel in the low nibble; an int8 weight code is the
byte (c < 0) << 7 | |c|.  Activation codes use the tensor-core operand
encoding: one byte (c < 0) << 7 | |c| per int4 code (e4m3 bits of c * 2^-9),
one 16-bit word (c < 0) << 15 | |c| per int8 code (f16 bits of c * 2^-24).
Asymmetric uint4 codes (W4A16) are unsigned nibbles,
eight channels per little-endian 32-bit word: channel 2i in bits [4i, 4i+4),
channel 2i+1 in bits [16+4i, 16+4i+4).
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# bf16 helpers (storage format of activations, weights, outputs, W4A16 scales)
# ----------------------------------------------------------------------------


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_round(x) -> np.ndarray:
    """float64 -> bf16 bit patterns, one rounding to nearest, ties to even.

    A bf16 number has 8 significant bits and the float32 exponent range, so
    a normal value a = m * 2^e (m in [0.5, 1)) is rounded on the grid
    2^(e-8); below the smallest normal (2^-126) the grid is fixed at 2^-133.
    Values that round past the largest finite bf16 become infinity.
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    _, e = np.frexp(a)
    quantum_exp = np.maximum(e - 8, -133)
    r = np.rint(np.ldexp(a, -quantum_exp))
    v = np.ldexp(r, quantum_exp)
    with np.errstate(over="ignore"):
        v32 = v.astype(np.float32)  # exact: v is on the bf16 grid (or overflows)
    bits = (v32.view(np.uint32) >> 16).astype(np.uint16)
    return np.where(neg, bits | np.uint16(0x8000), bits).astype(np.uint16)


def bf16_round_up_f32(v) -> np.ndarray:
    """Positive float32 -> the smallest bf16 value >= v, as float32 (R6)."""
    a = np.asarray(v, dtype=np.float32).astype(np.float64)
    _, e = np.frexp(a)
    quantum_exp = np.maximum(e - 8, -133)
    up = np.ldexp(np.ceil(np.ldexp(a, -quantum_exp)), quantum_exp)
    return up.astype(np.float32)


# ----------------------------------------------------------------------------
# Hadamard rotation (R1, R2)
# ----------------------------------------------------------------------------


def sylvester_hadamard(b: int) -> np.ndarray:
    """Unnormalised Sylvester Hadamard matrix H_b (int64, entries +-1).

    H_1 = [1];  H_2n = [[H_n, H_n], [H_n, -H_n]].
    """
    if b < 1 or (b & (b - 1)) != 0:
        raise ValueError("Hadamard size must be a power of two")
    H = np.ones((1, 1), dtype=np.int64)
    while H.shape[0] < b:
        H = np.block([[H, H], [H, -H]])
    return H


def block_hadamard_rotate(V, b: int) -> np.ndarray:
    """x~ = x . blockdiag(H_b / sqrt(b)) over the last axis, in float64.

    Written as (x . H_b) / sqrt(b): the +-1 products and their sums are exact
    in float64 for bf16 inputs, so the only rounding is the final division.
    """
    V = np.asarray(V, dtype=np.float64)
    if b == 0:
        return V.copy()
    R, K = V.shape
    if K % b:
        raise ValueError("K must be a multiple of the Hadamard block")
    H = sylvester_hadamard(b).astype(np.float64)
    blocks = V.reshape(R, K // b, b)
    out = np.matmul(blocks, H) / np.sqrt(np.float64(b))
    return out.reshape(R, K)


# ----------------------------------------------------------------------------
# Round-to-nearest quantizers (R3-R6)
# ----------------------------------------------------------------------------


def qmax_of(bits: int) -> int:
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    return (1 << (bits - 1)) - 1


def rtn_symmetric_rows(V32, bits: int):
    """Per-row symmetric RTN of float32 values.

    s = absmax / qmax (float32 division);  q = clamp(rint(v / s), -qmax, qmax).
    A row whose absmax is 0 gets s = 0 and all codes 0 (R5).
    """
    V32 = np.asarray(V32, dtype=np.float32)
    qmax = qmax_of(bits)
    absmax = np.max(np.abs(V32), axis=1)
    s = (absmax / np.float32(qmax)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = np.rint(V32 / safe[:, None])
    q = np.clip(q, -qmax, qmax)
    q = np.where(s[:, None] > 0, q, 0.0)
    return q.astype(np.int8), s


def rtn_static(V32, bits: int, scale: float):
    """Quantize with a given float32 scale: clamp(rint(v / s), -qmax, qmax)."""
    qmax = qmax_of(bits)
    s = np.float32(scale)
    if not s > 0:
        return np.zeros(np.shape(V32), dtype=np.int8)
    q = np.rint(np.asarray(V32, dtype=np.float32) / s)
    return np.clip(q, -qmax, qmax).astype(np.int8)


def rtn_asymmetric_groups(V32, group_size: int):
    """Asymmetric uint4 RTN over groups of `group_size` consecutive channels.

    lo = min(0, min v), hi = max(0, max v)           (float32)
    s  = bf16_round_up((hi - lo) / 15)                (float32 ops)
    z  = clamp(rint(-lo / s), 0, 15)
    q  = clamp(rint(v / s) + z, 0, 15)
    An all-zero group gets s = 1, z = 0 (R5).  Returns (q uint8 [R,K],
    s float32 [R,G], z float32 [R,G]); s and z are exact bf16 values.
    """
    V32 = np.asarray(V32, dtype=np.float32)
    R, K = V32.shape
    if K % group_size:
        raise ValueError("K must be a multiple of the group size")
    G = K // group_size
    Vg = V32.reshape(R, G, group_size)
    lo = np.minimum(np.float32(0), Vg.min(axis=2))
    hi = np.maximum(np.float32(0), Vg.max(axis=2))
    span = (hi - lo).astype(np.float32)
    s = bf16_round_up_f32((span / np.float32(15)).astype(np.float32))
    zero_group = span == 0
    s = np.where(zero_group, np.float32(1.0), s).astype(np.float32)
    z = np.clip(np.rint((-lo).astype(np.float32) / s), 0, 15).astype(np.float32)
    z = np.where(zero_group, np.float32(0.0), z).astype(np.float32)
    q = np.rint(Vg / s[:, :, None]) + z[:, :, None]
    q = np.clip(q, 0, 15).astype(np.uint8).reshape(R, K)
    return q, s, z


def quantize_weights_rtn(W_bits, bits: int, symmetric: bool, group_size: int = 0,
                         hadamard_block: int = 0):
    """Offline weight preparation (RTN, optional rotation folded into W).

    symmetric: W~ = W . blockdiag(H_b/sqrt(b)) (if b > 0), rounded to float32,
               then per-output-channel RTN; returns dict(q int8 [N,K], s [N]).
    asymmetric (bits = 4, group_size > 0, no rotation): per-group uint4 RTN;
               returns dict(q uint8 [N,K], s [N,G], z [N,G]).
    """
    W = bf16_to_f64(W_bits)
    if symmetric:
        if group_size != 0:
            raise ValueError("symmetric weights are per output channel")
        Wt32 = block_hadamard_rotate(W, hadamard_block).astype(np.float32)
        q, s = rtn_symmetric_rows(Wt32, bits)
        return dict(q=q, s=s)
    if bits != 4 or group_size <= 0 or hadamard_block != 0:
        raise ValueError("asymmetric weights are int4, group-wise, unrotated")
    q, s, z = rtn_asymmetric_groups(W.astype(np.float32), group_size)
    return dict(q=q, s=s, z=z)


def act_hadamard_quant(X_bits, bits: int, hadamard_block: int, static_scale=None):
    """Online activation rotation + per-token quantization.

    x~ = x . blockdiag(H_b/sqrt(b)) in float64, rounded to float32; then
    dynamic: s[m] = max_k |x~[m,k]| / qmax, codes by rtn_symmetric_rows;
    static:  s[m] = the given scale for every token, codes clamp to range.
    Returns (codes int8 [M,K], scales float32 [M]).
    """
    X = bf16_to_f64(X_bits)
    Xt32 = block_hadamard_rotate(X, hadamard_block).astype(np.float32)
    if static_scale is None:
        return rtn_symmetric_rows(Xt32, bits)
    q = rtn_static(Xt32, bits, static_scale)
    return q, np.full(X.shape[0], np.float32(static_scale), dtype=np.float32)


def rotated_f64(X_bits, hadamard_block: int) -> np.ndarray:
    """The exact-as-float64 rotated values (used to locate rounding ties)."""
    return block_hadamard_rotate(bf16_to_f64(X_bits), hadamard_block)


# ----------------------------------------------------------------------------
# Packing of codes (format definition)
# ----------------------------------------------------------------------------


def pack_int4(codes) -> np.ndarray:
    """[R, K] int4 codes in [-7, 7] -> [R, K/2] sign-magnitude bytes.

    Nibble of code c: (c < 0) << 3 | |c|; the even channel is the low nibble.
    """
    c = np.asarray(codes).astype(np.int64)
    if np.any(np.abs(c) > 7):
        raise ValueError("int4 codes must lie in [-7, 7]")
    nib = np.where(c < 0, 8, 0) | np.abs(c)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


def pack_uint4(codes) -> np.ndarray:
    """[R, K] asymmetric codes in [0, 15] -> [R, K/2] bytes (W4A16 layout).

    Each run of 8 channels is one little-endian 32-bit word: channel 2i in
    bits [4i, 4i+4), channel 2i+1 in bits [16+4i, 16+4i+4), i = 0..3.
    """
    c = np.asarray(codes).astype(np.int64)
    if np.any((c < 0) | (c > 15)):
        raise ValueError("uint4 codes must lie in [0, 15]")
    R, K = c.shape
    if K % 8:
        raise ValueError("K must be a multiple of 8")
    g = c.reshape(R, K // 8, 8)
    word = np.zeros((R, K // 8), dtype=np.int64)
    for i in range(4):
        word |= g[:, :, 2 * i] << (4 * i)
        word |= g[:, :, 2 * i + 1] << (16 + 4 * i)
    return word.astype("<u4").view(np.uint8).reshape(R, K // 2)


def unpack_uint4(packed) -> np.ndarray:
    """Inverse of pack_uint4."""
    p = np.ascontiguousarray(np.asarray(packed, dtype=np.uint8))
    R = p.shape[0]
    word = p.reshape(R, -1).view("<u4").astype(np.int64)
    out = np.empty((R, word.shape[1], 8), dtype=np.int64)
    for i in range(4):
        out[:, :, 2 * i] = (word >> (4 * i)) & 0xF
        out[:, :, 2 * i + 1] = (word >> (16 + 4 * i)) & 0xF
    return out.reshape(R, -1).astype(np.uint8)


def unpack_int4(packed, signed: bool = True) -> np.ndarray:
    """Inverse of pack_int4 (signed); plain nibbles when signed is False."""
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    lo, hi = p & 0xF, p >> 4
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.int64)
    out[:, 0::2], out[:, 1::2] = lo, hi
    if signed:
        out = np.where(out & 8, -(out & 7), out & 7)
    return out.astype(np.int8 if signed else np.uint8)


def pack_int8(codes) -> np.ndarray:
    """[R, K] int8 codes in [-127, 127] -> [R, K] sign-magnitude bytes."""
    c = np.asarray(codes).astype(np.int64)
    if np.any(np.abs(c) > 127):
        raise ValueError("int8 codes must lie in [-127, 127]")
    return (np.where(c < 0, 0x80, 0) | np.abs(c)).astype(np.uint8)


def unpack_int8(packed) -> np.ndarray:
    """Inverse of pack_int8."""
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    return np.where(p & 0x80, -(p & 0x7F), p & 0x7F).astype(np.int8)


def encode_act_int4(codes) -> np.ndarray:
    """[M, K] int4 activation codes in [-7, 7] -> [M, K] bytes (c < 0) << 7 | |c|.

    The byte is the e4m3 encoding of c * 2^-9 (a subnormal), which the
    integer GEMM feeds to the tensor cores unchanged.
    """
    c = np.asarray(codes).astype(np.int64)
    if np.any(np.abs(c) > 7):
        raise ValueError("int4 codes must lie in [-7, 7]")
    return (np.where(c < 0, 0x80, 0) | np.abs(c)).astype(np.uint8)


def decode_act_int4(enc) -> np.ndarray:
    e = np.asarray(enc, dtype=np.uint8).astype(np.int64)
    return np.where(e & 0x80, -(e & 0x7F), e & 0x7F).astype(np.int8)


def encode_act_int8(codes) -> np.ndarray:
    """[M, K] int8 activation codes in [-127, 127] -> [M, K] uint16 (c < 0) << 15 | |c|.

    The word is the f16 encoding of c * 2^-24 (a subnormal).
    """
    c = np.asarray(codes).astype(np.int64)
    if np.any(np.abs(c) > 127):
        raise ValueError("int8 codes must lie in [-127, 127]")
    return (np.where(c < 0, 0x8000, 0) | np.abs(c)).astype(np.uint16)


def decode_act_int8(enc) -> np.ndarray:
    e = np.asarray(enc).astype(np.int64) & 0xFFFF
    return np.where(e & 0x8000, -(e & 0x7FFF), e & 0x7FFF).astype(np.int16)


# ----------------------------------------------------------------------------
# Integer GEMM and epilogue
# ----------------------------------------------------------------------------


def int_gemm(xq, wq) -> np.ndarray:
    """acc[m, n] = sum_k xq[m, k] * wq[n, k], exact (int64).

    Evaluated with a float64 matrix product: every product and partial sum
    is an integer below 2^53 in magnitude (|code| <= 128, K < 2^30), where
    float64 arithmetic is exact whatever the summation order.
    """
    xq = np.asarray(xq)
    wq = np.asarray(wq)
    K = xq.shape[1]
    bound = int(np.abs(xq.astype(np.int64)).max(initial=0)) * \
        int(np.abs(wq.astype(np.int64)).max(initial=0)) * K
    if bound >= 2 ** 53:
        raise ValueError("integer GEMM outside the exact float64 range")
    acc = xq.astype(np.float64) @ wq.astype(np.float64).T
    return acc.astype(np.int64)


def linear_epilogue(acc, sx, sw, bias_bits=None) -> np.ndarray:
    """y = bf16(acc * s_x[m] * s_w[n] + bias[n]), evaluated in float64."""
    y = np.asarray(acc, dtype=np.float64) * np.asarray(sx, np.float64)[:, None] \
        * np.asarray(sw, np.float64)[None, :]
    if bias_bits is not None:
        y = y + bf16_to_f64(bias_bits)[None, :]
    return bf16_round(y)


def linear_quantized(X_bits, W_bits, bits: int, hadamard_block: int,
                     bias_bits=None, static_scale=None, act_bits=None):
    """Whole W4A4 / W8A8 projection from bf16 inputs to bf16 output; with
    act_bits = 8 and bits = 4, the W4A8 projection (int4 weights, int8
    per-token activations: the QuantVLA setting, "W4A8" in its results).

    Returns dict with the activation codes/scales, weight codes/scales, the
    int64 accumulators and the bf16 output bits.
    """
    wt = quantize_weights_rtn(W_bits, bits, True, 0, hadamard_block)
    xq, sx = act_hadamard_quant(X_bits, bits if act_bits is None else act_bits, hadamard_block, static_scale)
    acc = int_gemm(xq, wt["q"])
    y = linear_epilogue(acc, sx, wt["s"], bias_bits)
    return dict(xq=xq, sx=sx, wq=wt["q"], sw=wt["s"], acc=acc, y=y)


# ----------------------------------------------------------------------------
# Weight-only int4 (W4A16) and the bf16 reference
# ----------------------------------------------------------------------------


def dequant_w4a16(q, s, z, group_size: int) -> np.ndarray:
    """Wdq[n, k] = (q[n, k] - z[n, g]) * s[n, g], g = k // group_size (float32, exact)."""
    q = np.asarray(q, dtype=np.float32)
    N, K = q.shape
    G = K // group_size
    sg = np.repeat(np.asarray(s, np.float32).reshape(N, G), group_size, axis=1)
    zg = np.repeat(np.asarray(z, np.float32).reshape(N, G), group_size, axis=1)
    return ((q - zg) * sg).astype(np.float32)


def linear_w4a16(X_bits, q, s, z, group_size: int, bias_bits=None) -> np.ndarray:
    """y = bf16(sum_k x[m, k] * Wdq[n, k] (+ bias[n])), the sum in float64."""
    Wdq = dequant_w4a16(q, s, z, group_size).astype(np.float64)
    y = bf16_to_f64(X_bits) @ Wdq.T
    if bias_bits is not None:
        y = y + bf16_to_f64(bias_bits)[None, :]
    return bf16_round(y)


def linear_bf16(X_bits, W_bits, bias_bits=None) -> np.ndarray:
    """The 16-bit baseline: y = bf16(x . W^T (+ bias)), the sum in float64."""
    y = bf16_to_f64(X_bits) @ bf16_to_f64(W_bits).T
    if bias_bits is not None:
        y = y + bf16_to_f64(bias_bits)[None, :]
    return bf16_round(y)


# ----------------------------------------------------------------------------
# Static per-step activation scales (reduced per-step table, reading R9)
# ----------------------------------------------------------------------------


def calibrate_static_scale(X_bits_list, bits: int, hadamard_block: int) -> np.float32:
    """s = max over calibration draws and tokens of max|x~| / qmax (float32)."""
    qmax = qmax_of(bits)
    absmax = np.float32(0.0)
    for Xb in X_bits_list:
        Xt32 = block_hadamard_rotate(bf16_to_f64(Xb), hadamard_block).astype(np.float32)
        absmax = max(absmax, np.float32(np.max(np.abs(Xt32))))
    return np.float32(absmax / np.float32(qmax))
