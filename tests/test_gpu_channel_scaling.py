"""Channel scaling on the GPU (FoldQuantVLA abstract: channel scaling combined
with block Hadamard transforms and dynamic per-token quantization), against
oracle/scale_folding.py: W' = W diag(c) quantized offline, x' = x diag(1/c)
rotated and quantized online, the integer GEMM unchanged.

Bars: weight codes equal to the oracle's but where float64 rounding puts the
rotated value on the other side of a float32 rounding point next to a tie
(at most 1e-5 of codes, off by one); activation codes equal except within
1e-4 of a rounding tie of the exact quotient (at most 1e-4 of codes); the
projection within relative Frobenius error 1e-3 of linear_quantized_scaled.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_ptq_linear_vqlin_b300 as vq  # noqa: E402
from oracle import scale_folding as sf  # noqa: E402
from oracle import vqlin_oracle as o  # noqa: E402
from synth import activations, sub_rng, weights  # noqa: E402

DEV = torch.device("cuda:0")


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def bf16_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def channel_factors(Xb, K, seed):
    """A smoothing-style c: larger on the outlier channels (their per-channel
    absmax to the power 1/2), random elsewhere, positive float32."""
    amax = np.abs(o.bf16_to_f64(Xb)).max(axis=0)
    c = np.sqrt(np.maximum(amax, 1e-3)) * sub_rng(seed, "c", K).uniform(0.8, 1.25, K)
    return c.astype(np.float32)


def _case(M, N, K, seed):
    Xb = activations(M, K, n_outliers=max(1, K // 100), outlier_scale=40, seed=seed, tags=("cs", M, K))
    Wb = weights(N, K, seed=seed + 1, tags=("cs", N, K))
    return Xb, Wb, channel_factors(Xb, K, seed + 2)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("hb", [0, 64, 128])
def test_channel_scaled_codes(bits, hb):
    M, N, K = 33, 320, 2048
    Xb, Wb, c = _case(M, N, K, 201)
    cd = torch.from_numpy(c).to(DEV)
    wq, sw = vq.quantize_weights_rtn(to_dev_bf16(Wb), bits, True, 0, hb, channel_scale=cd)
    xq, sx = vq.act_hadamard_quant(to_dev_bf16(Xb), bits, hb, channel_scale=cd)
    vq.get_last_device_error()
    c64 = c.astype(np.float64)
    Wt = o.block_hadamard_rotate(o.bf16_to_f64(Wb) * c64[None, :], hb).astype(np.float32)
    wq_ref, sw_ref = o.rtn_symmetric_rows(Wt, bits)
    np.testing.assert_allclose(sw.cpu().numpy(), sw_ref, rtol=1e-6, atol=0)
    wcodes = wq.cpu().numpy().view(np.uint8)
    wcodes = o.unpack_int4(wcodes, signed=True) if bits == 4 else o.unpack_int8(wcodes)
    dw = wcodes.astype(np.int64) - wq_ref.astype(np.int64)
    assert np.abs(dw).max() <= 1 and np.count_nonzero(dw) <= max(1, int(1e-5 * dw.size))
    exact = o.block_hadamard_rotate(o.bf16_to_f64(Xb) / c64[None, :], hb)
    xq_ref, sx_ref = o.rtn_symmetric_rows(exact.astype(np.float32), bits)
    np.testing.assert_allclose(sx.cpu().numpy(), sx_ref, rtol=1e-5, atol=0)
    qn = xq.cpu().numpy()
    xcodes = o.decode_act_int4(qn) if bits == 4 else o.decode_act_int8(qn.view(np.uint16))
    dx = xcodes.astype(np.int64) - xq_ref.astype(np.int64)
    bad = np.nonzero(dx)
    assert np.all(np.abs(dx) <= 1)
    quot = exact / np.where(sx_ref > 0, sx_ref, 1).astype(np.float64)[:, None]
    assert np.all(np.abs(quot[bad] - np.floor(quot[bad]) - 0.5) < 1e-4), "a code differs away from a tie"
    assert bad[0].size <= 1e-4 * dx.size


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("hb", [64, 128])
def test_channel_scaled_projection(bits, hb):
    M, N, K = 50, 512, 1024
    Xb, Wb, c = _case(M, N, K, 211)
    bias = weights(1, N, std=0.5, seed=213)[0]
    cd = torch.from_numpy(c).to(DEV)
    wq, sw = vq.quantize_weights_rtn(to_dev_bf16(Wb), bits, True, 0, hb, channel_scale=cd)
    xq, sx = vq.act_hadamard_quant(to_dev_bf16(Xb), bits, hb, channel_scale=cd)
    fn = vq.linear_w4a4 if bits == 4 else vq.linear_w8a8
    y = fn(xq, sx, wq, sw, to_dev_bf16(bias))
    vq.get_last_device_error()
    ref = sf.linear_quantized_scaled(Xb, Wb, bits, hb, c=c.astype(np.float64), bias_bits=bias)
    a, r = o.bf16_to_f64(bf16_bits(y)), o.bf16_to_f64(ref["y"])
    err = np.linalg.norm(a - r) / np.linalg.norm(r)
    assert err <= 1e-3, f"relative Frobenius error {err}"


def test_unit_channel_scale_is_the_plain_path():
    # c = 1: dividing by one is exact, so the codes equal the unscaled call's bit for bit
    M, K = 16, 1024
    Xb = activations(M, K, n_outliers=4, outlier_scale=20, seed=221)
    one = torch.ones(K, dtype=torch.float32, device=DEV)
    for bits in (4, 8):
        q1, s1 = vq.act_hadamard_quant(to_dev_bf16(Xb), bits, 128, channel_scale=one)
        q0, s0 = vq.act_hadamard_quant(to_dev_bf16(Xb), bits, 128)
        assert torch.equal(q1, q0) and torch.equal(s1, s0)


# (M, N, K, hb): one launch (quantized on chip, clusters of 8 and 16), the
# activation kernel + few-token GEMM at long K, and + throughput GEMM beyond
# 128 tokens
STATIC_SCALED = [(50, 1024, 1024, 128), (50, 3072, 1024, 64), (16, 256, 256, 64), (50, 1024, 4096, 128),
                 (300, 512, 1024, 128)]


@pytest.mark.parametrize("case", STATIC_SCALED, ids=lambda c: "%dx%dx%d-b%d" % c)
def test_static_scale_with_channel_scaling(case):
    # the static-scale projection with channel scaling: the same codes and Y as
    # the activation kernel (static scale, channel factors) + the W4A4 GEMM,
    # bit for bit, and within 1e-3 of the oracle
    M, N, K, hb = case
    Xb, Wb, c = _case(M, N, K, 231)
    cd = torch.from_numpy(c).to(DEV)
    c64 = c.astype(np.float64)
    s = np.float32(o.calibrate_static_scale([activations(M, K, n_outliers=max(1, K // 100), outlier_scale=40,
                                                         seed=234, tags=("cs", M, K))], 4, hb))
    st = torch.tensor([s], dtype=torch.float32, device=DEV)
    X = to_dev_bf16(Xb)
    wq, sw = vq.quantize_weights_rtn(to_dev_bf16(Wb), 4, True, 0, hb, channel_scale=cd)
    xq = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    y = vq.linear_w4a4_static(X, st, wq, sw, hb, xq_out=xq, channel_scale=cd)
    vq.get_last_device_error()
    xq2, sx2 = vq.act_hadamard_quant(X, 4, hb, static_scale=st, channel_scale=cd)
    np.testing.assert_array_equal(xq.cpu().numpy(), xq2.cpu().numpy())
    np.testing.assert_array_equal(bf16_bits(y), bf16_bits(vq.linear_w4a4(xq2, sx2, wq, sw)))
    ref = sf.linear_quantized_scaled(Xb, Wb, 4, hb, c=c64, static_scale=s)
    a, r = o.bf16_to_f64(bf16_bits(y)), o.bf16_to_f64(ref["y"])
    assert np.linalg.norm(a - r) / np.linalg.norm(r) <= 1e-3
