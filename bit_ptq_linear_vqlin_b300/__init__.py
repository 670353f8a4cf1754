"""B300-native quantized linear projections (W4A4, W8A8, W4A16) for VLA PTQ.

Thin Python binding over libvqlin.so.  Every function here only marshals
arguments (device pointers, sizes, the current CUDA stream) and allocates
output tensors with PyTorch; all arithmetic runs in the library's CUDA
kernels.  The library has no CPU fallback: importing this package without
the built library, or calling it on CPU tensors, raises.

Tensor conventions (see include/vqlin.h):
  * activations X [M, K] and weights W [N, K] are torch.bfloat16, row-major;
  * symmetric codes lie in [-qmax, qmax] and are sign-magnitude: weight
    codes are torch.uint8, int4 [N, K/2] (nibble (c < 0) << 3 | |c|, even
    channel in the low nibble) or int8 [N, K] (byte (c < 0) << 7 | |c|);
    activation codes are in the tensor-core operand encoding, int4 as
    torch.uint8 [M, K] (byte (c < 0) << 7 | |c|) and int8 as torch.int16
    [M, K] (bits (c < 0) << 15 | |c|);
  * per-token / per-channel scales are float32; W4A16 group scales and zero
    points are bfloat16 [N, K/group].
"""
from __future__ import annotations

import ctypes

import torch

from ._abi import LIB_PATH, VqlinError, check, load  # noqa: F401

__all__ = [
    "VqlinError", "load", "LIB_PATH",
    "quantize_weights_rtn", "act_hadamard_quant", "linear_w4a4", "linear_w4a4_static", "linear_w8a8",
    "linear_w4a8", "linear_w4a16", "linear_bf16_ref", "debug_gemm_s32", "debug_gemm_w4a8_s32",
    "debug_gemm_withheld_loads", "debug_w4a16_withheld_loads", "measure_mma_rate",
    "composite_rotation_prepare", "quantize_weights_composite", "act_composite_quant",
    "init", "shutdown", "kernel_launch_count", "act_adaln_hadamard_quant",
    "get_last_device_error",
]

_lib = load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libvqlin has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def init() -> None:
    """Create the library's per-device state now (status word, cuBLASLt handle
    and workspace) instead of on first use."""
    check(_lib.vqlin_init(), "vqlin_init")


def shutdown() -> None:
    """Release the library's per-device state (after each device's queued work)."""
    check(_lib.vqlin_shutdown(), "vqlin_shutdown")


def kernel_launch_count() -> int:
    """The library's own kernel launches since it was loaded (graph replays not included)."""
    n = ctypes.c_ulonglong(0)
    check(_lib.vqlin_kernel_launch_count(ctypes.byref(n)), "vqlin_kernel_launch_count")
    return int(n.value)


def get_last_device_error(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded a device error."""
    check(_lib.vqlin_get_last_device_error(_stream(stream)), "vqlin_get_last_device_error")


def quantize_weights_rtn(W, bits: int, symmetric: bool = True, group_size: int = 0,
                         hadamard_block: int = 0, stream=None, channel_scale=None):
    """Offline RTN of W [N, K] bf16.  Returns (q, s) or, asymmetric, (q, s, z).
    channel_scale (float32 [K], symmetric only): quantize W . diag(c)."""
    _need(W, "W", torch.bfloat16, 2)
    N, K = W.shape
    dev = W.device
    if channel_scale is not None:
        if not symmetric:
            raise ValueError("channel scaling applies to the symmetric (rotated) weights")
        _need(channel_scale, "channel_scale", torch.float32, 1)
        q = torch.empty((N, K // 2) if bits == 4 else (N, K), dtype=torch.uint8, device=dev)
        s = torch.empty((N,), dtype=torch.float32, device=dev)
        check(_lib.vqlin_quantize_weights_rtn_scaled(_ptr(W), N, K, bits, hadamard_block, _ptr(channel_scale),
                                                     _ptr(q), _ptr(s), _stream(stream)),
              "vqlin_quantize_weights_rtn_scaled")
        return q, s
    q = torch.empty((N, K // 2) if bits == 4 else (N, K), dtype=torch.uint8, device=dev)
    if symmetric:
        s = torch.empty((N,), dtype=torch.float32, device=dev)
        z = None
    else:
        G = K // group_size if group_size > 0 else 0
        s = torch.empty((N, G), dtype=torch.bfloat16, device=dev)
        z = torch.empty((N, G), dtype=torch.bfloat16, device=dev)
    check(_lib.vqlin_quantize_weights_rtn(_ptr(W), N, K, bits, int(symmetric), group_size,
                                          hadamard_block, _ptr(q), _ptr(s), _ptr(z), _stream(stream)),
          "vqlin_quantize_weights_rtn")
    return (q, s) if symmetric else (q, s, z)


def act_hadamard_quant(X, bits: int, hadamard_block: int, static_scale=None, q_out=None,
                       scale_out=None, stream=None, channel_scale=None):
    """Rotate X [M, K] bf16 block-wise and quantize per token.  Returns (q, s).
    channel_scale (float32 [K]): rotate and quantize X . diag(1/c)."""
    _need(X, "X", torch.bfloat16, 2)
    M, K = X.shape
    if q_out is None:
        q_out = torch.empty((M, K), dtype=torch.uint8 if bits == 4 else torch.int16, device=X.device)
    if scale_out is None:
        scale_out = torch.empty((M,), dtype=torch.float32, device=X.device)
    if static_scale is not None:
        _need(static_scale, "static_scale", torch.float32)
    if channel_scale is not None:
        _need(channel_scale, "channel_scale", torch.float32, 1)
        check(_lib.vqlin_act_hadamard_quant_scaled(_ptr(X), M, K, bits, hadamard_block, _ptr(channel_scale),
                                                   _ptr(static_scale), _ptr(q_out), _ptr(scale_out),
                                                   _stream(stream)),
              "vqlin_act_hadamard_quant_scaled")
        return q_out, scale_out
    check(_lib.vqlin_act_hadamard_quant(_ptr(X), M, K, bits, hadamard_block, _ptr(static_scale),
                                        _ptr(q_out), _ptr(scale_out), _stream(stream)),
          "vqlin_act_hadamard_quant")
    return q_out, scale_out


def act_adaln_hadamard_quant(X, bits: int, hadamard_block: int, ada_scale, ada_shift, eps: float = 1e-6,
                             static_scale=None, q_out=None, scale_out=None, stream=None):
    """AdaLayerNorm of X [M, K] bf16 (per token, then (1 + ada_scale) and
    ada_shift per channel), rotated block-wise and quantized per token, in one
    kernel.  Returns (q, s) in the encoding of act_hadamard_quant."""
    _need(X, "X", torch.bfloat16, 2)
    _need(ada_scale, "ada_scale", torch.float32, 1)
    _need(ada_shift, "ada_shift", torch.float32, 1)
    M, K = X.shape
    if q_out is None:
        q_out = torch.empty((M, K), dtype=torch.uint8 if bits == 4 else torch.int16, device=X.device)
    if scale_out is None:
        scale_out = torch.empty((M,), dtype=torch.float32, device=X.device)
    if static_scale is not None:
        _need(static_scale, "static_scale", torch.float32)
    check(_lib.vqlin_act_adaln_hadamard_quant(_ptr(X), M, K, bits, hadamard_block, _ptr(ada_scale), _ptr(ada_shift),
                                              float(eps), _ptr(static_scale), _ptr(q_out), _ptr(scale_out),
                                              _stream(stream)),
          "vqlin_act_adaln_hadamard_quant")
    return q_out, scale_out


def composite_rotation_prepare(W, block: int, stream=None):
    """Offline: the zig-zag permutation and block rotations R_j = V_j H_b / sqrt(b)
    of W [N, K] bf16.  Returns (perm int32 [K], R float64 [K/b, b, b])."""
    _need(W, "W", torch.bfloat16, 2)
    N, K = W.shape
    perm = torch.empty((K,), dtype=torch.int32, device=W.device)
    R = torch.empty((K // block, block, block), dtype=torch.float64, device=W.device)
    check(_lib.vqlin_composite_rotation_prepare(_ptr(W), N, K, block, _ptr(perm), _ptr(R), _stream(stream)),
          "vqlin_composite_rotation_prepare")
    return perm, R


def quantize_weights_composite(W, bits: int, block: int, perm, R, stream=None):
    """Offline: W[:, perm] . blockdiag(R_j), per-output-channel symmetric RTN.
    Returns (q, s) in the layout of quantize_weights_rtn."""
    _need(W, "W", torch.bfloat16, 2)
    _need(perm, "perm", torch.int32, 1)
    _need(R, "R", torch.float64, 3)
    N, K = W.shape
    q = torch.empty((N, K // 2) if bits == 4 else (N, K), dtype=torch.uint8, device=W.device)
    s = torch.empty((N,), dtype=torch.float32, device=W.device)
    check(_lib.vqlin_quantize_weights_composite(_ptr(W), N, K, bits, block, _ptr(perm), _ptr(R), _ptr(q), _ptr(s),
                                                _stream(stream)),
          "vqlin_quantize_weights_composite")
    return q, s


def act_composite_quant(X, bits: int, block: int, perm, R, q_out=None, scale_out=None, stream=None):
    """Online: X[:, perm] . blockdiag(R_j), per-token dynamic quantization.
    Returns (q, s) in the encoding of act_hadamard_quant."""
    _need(X, "X", torch.bfloat16, 2)
    _need(perm, "perm", torch.int32, 1)
    _need(R, "R", torch.float64, 3)
    M, K = X.shape
    if q_out is None:
        q_out = torch.empty((M, K), dtype=torch.uint8 if bits == 4 else torch.int16, device=X.device)
    if scale_out is None:
        scale_out = torch.empty((M,), dtype=torch.float32, device=X.device)
    check(_lib.vqlin_act_composite_quant(_ptr(X), M, K, bits, block, _ptr(perm), _ptr(R), _ptr(q_out),
                                         _ptr(scale_out), _stream(stream)),
          "vqlin_act_composite_quant")
    return q_out, scale_out


def _linear_int(fn, what, xq, sx, wq, sw, bias, out, K, stream):
    M, N = xq.shape[0], wq.shape[0]
    _need(sx, "sx", torch.float32, 1)
    _need(sw, "sw", torch.float32, 1)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, 1)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    check(fn(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw), _ptr(bias), _ptr(out), M, N, K,
             _stream(stream)), what)
    return out


def linear_w4a4(xq, sx, wq, sw, bias=None, out=None, stream=None):
    """Y = bf16(int_gemm(xq, wq) * sx * sw + bias): xq uint8 [M, K], wq uint8 [N, K/2]."""
    _need(xq, "xq", torch.uint8, 2)
    _need(wq, "wq", torch.uint8, 2)
    if wq.shape[1] * 2 != xq.shape[1]:
        raise ValueError("wq must be [N, K/2] for xq [M, K]")
    return _linear_int(_lib.vqlin_linear_w4a4, "vqlin_linear_w4a4", xq, sx, wq, sw, bias, out,
                       xq.shape[1], stream)


def linear_w4a4_static(X, static_scale, wq, sw, hadamard_block: int = 128, bias=None, out=None,
                       xq_out=None, stream=None, channel_scale=None):
    """W4A4 with the activations quantized inside the GEMM at a static scale:
    the same Y as act_hadamard_quant(X, 4, hadamard_block, static_scale) followed
    by linear_w4a4.  X bf16 [M, K], static_scale float32 (one element), wq uint8
    [N, K/2].  xq_out (uint8 [M, K], allocated if None) receives the activation
    codes; the kernel also uses it to share them among its CTAs.
    channel_scale (float32 [K]): quantize X . diag(1/c) (wq from W . diag(c))."""
    _need(X, "X", torch.bfloat16, 2)
    _need(static_scale, "static_scale", torch.float32)
    _need(wq, "wq", torch.uint8, 2)
    _need(sw, "sw", torch.float32, 1)
    M, K = X.shape
    N = wq.shape[0]
    if wq.shape[1] * 2 != K:
        raise ValueError("wq must be [N, K/2] for X [M, K]")
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, 1)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    if xq_out is None:
        xq_out = torch.empty((M, K), dtype=torch.uint8, device=X.device)
    _need(xq_out, "xq_out", torch.uint8, 2)
    if tuple(xq_out.shape) != (M, K):
        raise ValueError("xq_out must be [M, K]")
    if channel_scale is not None:
        _need(channel_scale, "channel_scale", torch.float32, 1)
        check(_lib.vqlin_linear_w4a4_static_scaled(_ptr(X), _ptr(static_scale), _ptr(channel_scale), hadamard_block,
                                                   _ptr(wq), _ptr(sw), _ptr(bias), _ptr(out), _ptr(xq_out), M, N, K,
                                                   _stream(stream)),
              "vqlin_linear_w4a4_static_scaled")
        return out
    check(_lib.vqlin_linear_w4a4_static(_ptr(X), _ptr(static_scale), hadamard_block, _ptr(wq), _ptr(sw),
                                        _ptr(bias), _ptr(out), _ptr(xq_out), M, N, K, _stream(stream)),
          "vqlin_linear_w4a4_static")
    return out


def linear_w8a8(xq, sx, wq, sw, bias=None, out=None, stream=None):
    """Y = bf16(int_gemm(xq, wq) * sx * sw + bias): xq int16 [M, K], wq uint8 [N, K]."""
    _need(xq, "xq", torch.int16, 2)
    _need(wq, "wq", torch.uint8, 2)
    if wq.shape[1] != xq.shape[1]:
        raise ValueError("wq must be [N, K] for xq [M, K]")
    return _linear_int(_lib.vqlin_linear_w8a8, "vqlin_linear_w8a8", xq, sx, wq, sw, bias, out,
                       xq.shape[1], stream)


def linear_w4a8(xq, sx, wq, sw, bias=None, out=None, stream=None):
    """Y = bf16(int_gemm(xq, wq) * sx * sw + bias): xq int16 [M, K] (int8 activation
    codes), wq uint8 [N, K/2] (int4 weight codes)."""
    _need(xq, "xq", torch.int16, 2)
    _need(wq, "wq", torch.uint8, 2)
    if wq.shape[1] * 2 != xq.shape[1]:
        raise ValueError("wq must be [N, K/2] for xq [M, K]")
    return _linear_int(_lib.vqlin_linear_w4a8, "vqlin_linear_w4a8", xq, sx, wq, sw, bias, out,
                       xq.shape[1], stream)


def linear_w4a16(X, wq, scales, zeros, group_size: int = 128, bias=None, out=None, stream=None):
    """Y = bf16(X . dequant(wq, scales, zeros)^T + bias), weight-only int4."""
    _need(X, "X", torch.bfloat16, 2)
    _need(wq, "wq", torch.uint8, 2)
    _need(scales, "scales", torch.bfloat16, 2)
    _need(zeros, "zeros", torch.bfloat16, 2)
    M, K = X.shape
    N = wq.shape[0]
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, 1)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    check(_lib.vqlin_linear_w4a16(_ptr(X), _ptr(wq), _ptr(scales), _ptr(zeros), group_size,
                                  _ptr(bias), _ptr(out), M, N, K, _stream(stream)),
          "vqlin_linear_w4a16")
    return out


def linear_bf16_ref(X, W, bias=None, out=None, stream=None):
    """The 16-bit baseline Y = bf16(X . W^T + bias) (cuBLASLt)."""
    _need(X, "X", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 2)
    M, K = X.shape
    N = W.shape[0]
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, 1)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    check(_lib.vqlin_linear_bf16_ref(_ptr(X), _ptr(W), _ptr(bias), _ptr(out), M, N, K,
                                     _stream(stream)), "vqlin_linear_bf16_ref")
    return out


def debug_gemm_s32(bits: int, xq, wq, K: int, out=None, stream=None):
    """int32 accumulators of the W4A4 (bits 4) / W8A8 (bits 8) integer GEMM."""
    M, N = xq.shape[0], wq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=xq.device)
    check(_lib.vqlin_debug_gemm_s32(bits, _ptr(xq), _ptr(wq), _ptr(out), M, N, K, _stream(stream)),
          "vqlin_debug_gemm_s32")
    return out


def debug_gemm_w4a8_s32(xq, wq, K: int, out=None, stream=None):
    """int32 accumulators of the W4A8 integer GEMM (xq int16 [M, K], wq uint8 [N, K/2])."""
    M, N = xq.shape[0], wq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=xq.device)
    check(_lib.vqlin_debug_gemm_w4a8_s32(_ptr(xq), _ptr(wq), _ptr(out), M, N, K, _stream(stream)),
          "vqlin_debug_gemm_w4a8_s32")
    return out


def debug_gemm_withheld_loads(bits: int, xq, wq, K: int, limit_ns: int, out=None, stream=None):
    """Failure-detection test: launch the integer GEMM with every tile load
    withheld, so its bounded waits run out after limit_ns.  The error is then
    raised by get_last_device_error()."""
    M, N = xq.shape[0], wq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=xq.device)
    check(_lib.vqlin_debug_gemm_withheld_loads(bits, _ptr(xq), _ptr(wq), _ptr(out), M, N, K,
                                               ctypes.c_uint64(limit_ns), _stream(stream)),
          "vqlin_debug_gemm_withheld_loads")
    return out


def debug_w4a16_withheld_loads(X, wq, scales, zeros, group_size: int, limit_ns: int, out=None, stream=None):
    """Failure-detection hook: the W4A16 tensor-core kernel with every tile load
    withheld, so its bounded waits run out after limit_ns.  The error is then
    read with get_last_device_error()."""
    _need(X, "X", torch.bfloat16, 2)
    _need(wq, "wq", torch.uint8, 2)
    M, K = X.shape
    N = wq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    check(_lib.vqlin_debug_w4a16_withheld_loads(_ptr(X), _ptr(wq), _ptr(scales), _ptr(zeros), group_size,
                                                _ptr(out), M, N, K, limit_ns, _stream(stream)),
          "vqlin_debug_w4a16_withheld_loads")
    return out


def measure_mma_rate(kind: str, n: int, a_in_tmem: bool = True, accumulators: int = 1, issuers: int = 1,
                     iters: int = 4096, ctas=None, device=None, stream=None):
    """Dense rate of one tcgen05 MMA kind on this GPU ("e4m3": kind::f8f6f4,
    "bf16": kind::f16): (TFLOP/s over all CTAs, SM clocks per 128 x n x K MMA),
    with the MMAs spread over `accumulators` independent accumulators issued
    by `issuers` warps."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if ctas is None:
        ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.empty((ctas,), dtype=torch.int64, device=dev)
    tf, cpm = ctypes.c_double(0.0), ctypes.c_double(0.0)
    k = {"e4m3": 0, "bf16": 1}[kind]
    check(_lib.vqlin_measure_mma_rate(k, int(a_in_tmem), n, accumulators, issuers, iters, ctas, _ptr(cyc),
                                      ctypes.byref(tf),
                                      ctypes.byref(cpm), _stream(stream)), "vqlin_measure_mma_rate")
    return tf.value, cpm.value
