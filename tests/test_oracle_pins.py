"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against a closed form, an independent brute
force, an invariant of the mathematics, or a hand-derived fixture under
tests/golden/.  The pages print no worked numerical example, so no fixture
comes from them.
"""
import os

import numpy as np
import pytest

from oracle import vqlin_oracle as o
from synth import activations, weights, random_codes, f32_to_bf16_bits
from tests.conftest import GOLDEN


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]


# ---------------------------------------------------------------- Hadamard

@pytest.mark.parametrize("b", [1, 2, 4, 8, 16, 32, 64, 128])
def test_hadamard_rows_orthogonal_exactly(b):
    H = o.sylvester_hadamard(b)
    assert np.array_equal(H @ H.T, b * np.eye(b, dtype=np.int64))
    assert np.array_equal(H, H.T)


@pytest.mark.parametrize("b", [2, 8, 64, 128])
def test_hadamard_closed_form(b):
    # entry (i, j) of Sylvester's matrix is (-1)^popcount(i & j)
    H = o.sylvester_hadamard(b)
    for i in range(b):
        for j in range(b):
            assert H[i, j] == (-1) ** bin(i & j).count("1")


def test_hadamard_golden_h8():
    rows = [[int(v) for v in ln.split()] for ln in _golden_lines("hadamard_h8.txt")]
    assert np.array_equal(o.sylvester_hadamard(8), np.array(rows))


def _fwht_recursive(v):
    """Independent fast Walsh-Hadamard transform (unnormalised), by halves."""
    n = len(v)
    if n == 1:
        return [v[0]]
    a = _fwht_recursive(v[: n // 2])
    c = _fwht_recursive(v[n // 2:])
    return [x + y for x, y in zip(a, c)] + [x - y for x, y in zip(a, c)]


@pytest.mark.parametrize("b", [64, 128])
def test_rotation_matches_recursive_fwht(b):
    xb = activations(3, 2 * b, seed=5, tags=("fwht", b))
    x = o.bf16_to_f64(xb)
    got = o.block_hadamard_rotate(x, b)
    for r in range(3):
        for j in range(2):
            ref = np.array(_fwht_recursive(list(x[r, j * b:(j + 1) * b]))) / np.sqrt(b)
            np.testing.assert_allclose(got[r, j * b:(j + 1) * b], ref, rtol=0, atol=1e-14)


@pytest.mark.parametrize("b", [64, 128])
def test_rotation_of_one_hot_is_flat(b):
    K = 2 * b
    for c in (0, 5, b + 17, K - 1):
        x = np.zeros((1, K))
        x[0, c] = 3.0
        xt = o.block_hadamard_rotate(x, b)
        blk = c // b
        inside = xt[0, blk * b:(blk + 1) * b]
        np.testing.assert_allclose(np.abs(inside), 3.0 / np.sqrt(b), rtol=1e-15)
        signs = np.array([(-1) ** bin((c % b) & j).count("1") for j in range(b)])
        assert np.array_equal(np.sign(inside), signs)
        outside = np.delete(xt[0], np.arange(blk * b, (blk + 1) * b))
        assert np.all(outside == 0)


@pytest.mark.parametrize("b", [64, 128])
def test_rotation_is_an_involution(b):
    # H_b / sqrt(b) is symmetric and orthogonal, so applying it twice is identity
    x = o.bf16_to_f64(activations(4, 4 * b, seed=2, tags=("inv",)))
    back = o.block_hadamard_rotate(o.block_hadamard_rotate(x, b), b)
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-13 * np.abs(x).max())


@pytest.mark.parametrize("b", [64, 128])
def test_rotation_preserves_the_gemm(b):
    x = o.bf16_to_f64(activations(16, 512, n_outliers=4, outlier_scale=20, seed=3))
    w = o.bf16_to_f64(weights(32, 512, seed=3))
    y = x @ w.T
    yr = o.block_hadamard_rotate(x, b) @ o.block_hadamard_rotate(w, b).T
    assert np.linalg.norm(yr - y) / np.linalg.norm(y) < 1e-12


# ---------------------------------------------------------------- RTN

def test_rtn_golden_cases():
    for ln in _golden_lines("rtn_cases.txt"):
        bits, vals, scale, codes = [p.strip() for p in ln.split("|")]
        v = np.array([[float(t) for t in vals.split()]], dtype=np.float32)
        q, s = o.rtn_symmetric_rows(v, int(bits))
        assert s[0] == np.float32(float(scale))
        assert q[0].tolist() == [int(t) for t in codes.split()]


@pytest.mark.parametrize("bits", [4, 8])
def test_rtn_symmetric_invariants(bits):
    qmax = 7 if bits == 4 else 127
    v = o.bf16_to_f64(weights(64, 256, spike_frac=0.01, spike_scale=10, seed=9)).astype(np.float32)
    q, s = o.rtn_symmetric_rows(v, bits)
    assert q.min() >= -qmax and q.max() <= qmax
    err = np.abs(v.astype(np.float64) - q.astype(np.float64) * s[:, None].astype(np.float64))
    # half a step, plus the rounding of the float32 quotient v / s (R4)
    assert np.all(err <= s[:, None].astype(np.float64) / 2 + np.abs(v) * 2.0 ** -23)
    am = np.argmax(np.abs(v), axis=1)
    assert np.all(np.abs(q[np.arange(64), am]) == qmax)
    np.testing.assert_array_equal(s, (np.abs(v).max(axis=1) / np.float32(qmax)).astype(np.float32))


def test_rtn_static_clamps_beyond_range():
    v = np.array([[0.5, -0.5, 100.0, -100.0, 6.9, -7.6, 2.5]], dtype=np.float32)
    q = o.rtn_static(v, 4, 1.0)
    # symmetric range [-qmax, qmax]: -100 and -7.6 clamp to -7, not to -8
    assert q[0].tolist() == [0, 0, 7, -7, 7, -7, 2]
    q8 = o.rtn_static(v, 8, 0.5)
    assert q8[0].tolist() == [1, -1, 127, -127, 14, -15, 5]


def test_rtn_asymmetric_hand_cases():
    g = 8
    # range [0, 15]: s = 1, z = 0, q = rint(v)
    v = np.array([[0, 15, 1.5, 2.5, 7, 3, 14.5, 0.5]], dtype=np.float32)
    q, s, z = o.rtn_asymmetric_groups(v, g)
    assert s[0, 0] == 1 and z[0, 0] == 0
    assert q[0].tolist() == [0, 15, 2, 2, 7, 3, 14, 0]
    # range [-1, 14]: s = 1, z = 1, q = rint(v) + 1
    v = np.array([[-1, 14, 0, 2.5, -0.5, 3, 13.5, 6]], dtype=np.float32)
    q, s, z = o.rtn_asymmetric_groups(v, g)
    assert s[0, 0] == 1 and z[0, 0] == 1
    assert q[0].tolist() == [0, 15, 1, 3, 1, 4, 15, 7]
    # all positive: the range is widened to include 0, so z = 0
    v = np.array([[1, 2, 3, 4, 5, 6, 7, 30]], dtype=np.float32)
    q, s, z = o.rtn_asymmetric_groups(v, g)
    assert s[0, 0] == 2 and z[0, 0] == 0
    assert q[0].tolist() == [0, 1, 2, 2, 2, 3, 4, 15]
    # all zero: s = 1, z = 0
    q, s, z = o.rtn_asymmetric_groups(np.zeros((1, g), np.float32), g)
    assert s[0, 0] == 1 and z[0, 0] == 0 and q.max() == 0


def test_rtn_asymmetric_invariants():
    w = o.bf16_to_f64(weights(32, 512, spike_frac=0.001, spike_scale=10, seed=4)).astype(np.float32)
    q, s, z = o.rtn_asymmetric_groups(w, 128)
    assert q.min() >= 0 and q.max() <= 15
    assert np.array_equal(z, np.rint(z)) and z.min() >= 0 and z.max() <= 15
    # s is a bf16 value: its low 16 float32 bits are zero
    assert np.all((s.view(np.uint32) & 0xFFFF) == 0)
    wg = w.reshape(32, 4, 128).astype(np.float64)
    span = np.maximum(wg.max(axis=2), 0) - np.minimum(wg.min(axis=2), 0)
    assert np.all(15 * s.astype(np.float64) >= span * (1 - 2 ** -22))
    deq = (q.reshape(32, 4, 128).astype(np.float64) - z[:, :, None]) * s[:, :, None]
    assert np.all(np.abs(wg - deq) <= s[:, :, None] / 2 * (1 + 1e-6))


def test_bf16_round_golden():
    for ln in _golden_lines("bf16_round_cases.txt"):
        val, bits = ln.split()
        assert int(o.bf16_round(np.array([float(val)]))[0]) == int(bits, 16), val


def test_bf16_round_is_nearest():
    # brute force: the chosen bf16 is at least as close as both neighbours
    rng = np.random.default_rng(0)
    x = rng.standard_normal(2000) * 10.0 ** rng.integers(-5, 5, 2000)
    b = o.bf16_round(x).astype(np.int64)
    v = o.bf16_to_f64(b.astype(np.uint16))
    for nb in (b - 1, b + 1):
        vn = o.bf16_to_f64((nb & 0xFFFF).astype(np.uint16))
        assert np.all(np.abs(v - x) <= np.abs(vn - x))


# ---------------------------------------------------------------- integer GEMM

def _gemm_bruteforce(xq, wq):
    M, K = xq.shape
    N = wq.shape[0]
    out = [[0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = 0
            for k in range(K):
                acc += int(xq[m, k]) * int(wq[n, k])
            out[m][n] = acc
    return np.array(out, dtype=np.int64)


def _gemm_bruteforce_kouter(xq, wq):
    M, K = xq.shape
    out = np.zeros((M, wq.shape[0]), dtype=object)
    for k in range(K):
        out += np.outer(xq[:, k].astype(object), wq[:, k].astype(object))
    return out.astype(np.int64)


@pytest.mark.parametrize("bits", [4, 8])
def test_int_gemm_bruteforce(bits):
    lo, hi = (-7, 7) if bits == 4 else (-127, 127)
    xq = random_codes((5, 96), lo, hi, seed=1)
    wq = random_codes((7, 96), lo, hi, seed=2)
    ref = _gemm_bruteforce(xq, wq)
    assert np.array_equal(_gemm_bruteforce_kouter(xq, wq), ref)
    assert np.array_equal(o.int_gemm(xq, wq), ref)


def test_int_gemm_adversarial_extremes():
    K = 16384
    x = np.full((2, K), -7, np.int8)
    w = np.full((3, K), -7, np.int8)
    assert np.all(o.int_gemm(x, w) == 49 * K)
    x8 = np.full((2, K), -127, np.int8)
    w8 = np.full((2, K), -127, np.int8)
    w8[1, ::2] = 126
    acc = o.int_gemm(x8, w8)
    assert acc[0, 0] == 16129 * K and acc[0, 1] == (16129 - 127 * 126) * K // 2


def test_pack_int4_format():
    # sign-magnitude nibbles (c < 0) << 3 | |c|, even channel in the low nibble
    codes = np.array([[1, -1, -7, 7, 0, 5]], dtype=np.int8)
    p = o.pack_int4(codes)
    assert p[0].tolist() == [0x91, 0x7F, 0x50]
    assert np.array_equal(o.unpack_int4(p, True), codes)
    with pytest.raises(ValueError):
        o.pack_int4(np.array([[-8, 0]], dtype=np.int8))



def test_activation_code_encodings_are_exact_float_operands():
    # int4 activation code c -> byte (c < 0) << 7 | |c|, the e4m3 bits of
    # c * 2^-9 (exponent field 0: value (-1)^s * m * 2^-9); int8 -> 16-bit
    # (c < 0) << 15 | |c|, the f16 bits of c * 2^-24 (value (-1)^s * m * 2^-24)
    c4 = np.arange(-7, 8).reshape(1, -1)
    e4 = o.encode_act_int4(c4)
    assert e4[0].tolist()[:3] == [0x87, 0x86, 0x85] and e4[0, 7] == 0 and e4[0, 14] == 0x07
    sign = np.where(e4 & 0x80, -1.0, 1.0)
    assert np.array_equal(sign * (e4 & 0x07) * 2.0 ** -9, c4 * 2.0 ** -9)
    assert np.array_equal(o.decode_act_int4(e4), c4)
    c8 = np.array([[-127, -64, -1, 0, 1, 100, 127]])
    e8 = o.encode_act_int8(c8)
    assert e8[0].tolist() == [0x807F, 0x8040, 0x8001, 0, 1, 100, 127]
    assert np.array_equal(e8.view(np.float16).astype(np.float64), c8 * 2.0 ** -24)
    assert np.array_equal(o.decode_act_int8(e8), c8)
    with pytest.raises(ValueError):
        o.encode_act_int4(np.array([[8]]))


def test_pack_uint4_format():
    # one 32-bit little-endian word per 8 channels: channel 2i in bits
    # [4i, 4i+4), channel 2i+1 in bits [16+4i, 16+4i+4)
    u = np.array([[1, 2, 3, 4, 5, 6, 7, 8, 15, 0, 0, 0, 0, 0, 0, 9]], dtype=np.uint8)
    p = o.pack_uint4(u)
    # word 0: evens 1,3,5,7 -> 0x7531; odds 2,4,6,8 -> 0x8642
    # word 1: evens 15,0,0,0 -> 0x000F; odds 0,0,0,9 -> 0x9000
    assert p[0].tolist() == [0x31, 0x75, 0x42, 0x86, 0x0F, 0x00, 0x00, 0x90]
    assert np.array_equal(o.unpack_uint4(p), u)
    r = random_codes((3, 64), 0, 15, seed=3).astype(np.uint8)
    assert np.array_equal(o.unpack_uint4(o.pack_uint4(r)), r)
    with pytest.raises(ValueError):
        o.pack_uint4(np.array([[16] + [0] * 7]))


def test_pack_int8_format():
    codes = np.array([[1, -1, 127, -127, 0, -64]], dtype=np.int8)
    p = o.pack_int8(codes)
    assert p[0].tolist() == [0x01, 0x81, 0x7F, 0xFF, 0x00, 0xC0]
    assert np.array_equal(o.unpack_int8(p), codes)
    with pytest.raises(ValueError):
        o.pack_int8(np.array([[-128]], dtype=np.int16))


# ---------------------------------------------------------------- epilogue / W4A16 / bf16

def test_epilogue_unit_scales_is_bf16_of_acc():
    acc = np.array([[0, 1, -255, 256, 257, 259]], dtype=np.int64)
    y = o.linear_epilogue(acc, np.ones(1, np.float32), np.ones(6, np.float32))
    expect = [0x0000, 0x3F80, 0xC37F, 0x4380, 0x4380, 0x4382]
    assert y[0].tolist() == expect


def test_w4a16_reduces_to_integer_gemm():
    # s = 1 and z = 8 make Wdq = q - 8; integer activations make the output exact
    N, K, g = 6, 256, 128
    q = random_codes((N, K), 0, 15, seed=7).astype(np.uint8)
    xi = random_codes((3, K), -3, 3, seed=8)
    xb = f32_to_bf16_bits(xi.astype(np.float32))
    s = np.ones((N, K // g), np.float32)
    z = np.full((N, K // g), 8, np.float32)
    y = o.linear_w4a16(xb, q, s, z, g)
    ref = _gemm_bruteforce(xi, q.astype(np.int64) - 8)
    assert np.array_equal(o.bf16_to_f64(y), ref.astype(np.float64))  # |ref| < 256 is exact


def test_w4a16_dequant_bruteforce():
    N, K, g = 2, 256, 128
    q = random_codes((N, K), 0, 15, seed=11).astype(np.uint8)
    s = np.array([[0.5, 0.25], [0.125, 2.0]], np.float32)
    z = np.array([[3, 8], [15, 0]], np.float32)
    d = o.dequant_w4a16(q, s, z, g)
    for n in range(N):
        for k in range(K):
            assert d[n, k] == (int(q[n, k]) - z[n, k // g]) * s[n, k // g]


def test_linear_bf16_bruteforce():
    xb = activations(3, 32, seed=1)
    wb = weights(4, 32, seed=1)
    x, w = o.bf16_to_f64(xb), o.bf16_to_f64(wb)
    y = o.linear_bf16(xb, wb)
    for m in range(3):
        for n in range(4):
            exact = sum(x[m, k] * w[n, k] for k in range(32))
            assert y[m, n] == o.bf16_round(np.array([exact]))[0]


# ---------------------------------------------------------------- whole projection

@pytest.mark.parametrize("bits,b,abits", [(4, 64, 4), (4, 128, 4), (8, 128, 8), (4, 0, 4), (4, 128, 8)])
def test_quantized_linear_within_rtn_error_bound(bits, b, abits):
    """|y - x.W^T| <= sum_k (|x~| s_w/2 + |w~| s_x/2 + s_x s_w/4) + half a bf16 ulp."""
    M, N, K = 8, 16, 256
    xb = activations(M, K, n_outliers=4, outlier_scale=20, seed=21)
    wb = weights(N, K, seed=22)
    r = o.linear_quantized(xb, wb, bits, b, act_bits=abits)
    assert np.abs(r["xq"]).max() <= (7 if abits == 4 else 127) and np.abs(r["wq"]).max() <= (7 if bits == 4 else 127)
    x, w = o.bf16_to_f64(xb), o.bf16_to_f64(wb)
    exact = x @ w.T
    xt = np.abs(o.block_hadamard_rotate(x, b))
    wt = np.abs(o.block_hadamard_rotate(w, b))
    sx = r["sx"].astype(np.float64)[:, None]
    sw = r["sw"].astype(np.float64)[None, :]
    bound = (xt.sum(1)[:, None] * sw / 2 + wt.sum(1)[None, :] * sx / 2 + K * sx * sw / 4)
    bound = bound * (1 + 1e-5) + np.abs(exact) * 2.0 ** -8 + 1e-30
    y = o.bf16_to_f64(r["y"])
    assert np.all(np.abs(y - exact) <= bound)
    # and the float64 value of the accumulators is what the epilogue scales
    assert np.array_equal(r["acc"], _gemm_bruteforce_kouter(r["xq"], r["wq"]))


def test_rotation_reduces_w4a4_error_on_outlier_inputs():
    M, N, K = 32, 64, 512
    xb = activations(M, K, n_outliers=5, outlier_scale=20, seed=31)
    wb = weights(N, K, seed=32)
    exact = o.bf16_to_f64(xb) @ o.bf16_to_f64(wb).T
    e_plain = np.linalg.norm(o.bf16_to_f64(o.linear_quantized(xb, wb, 4, 0)["y"]) - exact)
    e_rot = np.linalg.norm(o.bf16_to_f64(o.linear_quantized(xb, wb, 4, 128)["y"]) - exact)
    assert e_rot < 0.5 * e_plain


def test_w4a8_sits_between_w4a4_and_w8a8():
    # 8-bit activations remove the activation part of the W4A4 error; 4-bit
    # weights keep the weight part that W8A8 does not have
    M, N, K = 32, 64, 512
    xb = activations(M, K, n_outliers=5, outlier_scale=20, seed=33)
    wb = weights(N, K, seed=34)
    exact = o.bf16_to_f64(xb) @ o.bf16_to_f64(wb).T
    err = {name: np.linalg.norm(o.bf16_to_f64(o.linear_quantized(xb, wb, wbits, 128, act_bits=abits)["y"]) - exact)
           for name, wbits, abits in (("w4a4", 4, 4), ("w4a8", 4, 8), ("w8a8", 8, 8))}
    assert err["w8a8"] < err["w4a8"] < err["w4a4"]
    # same weight codes as W4A4 and same activation codes as W8A8
    r48 = o.linear_quantized(xb, wb, 4, 128, act_bits=8)
    assert np.array_equal(r48["wq"], o.linear_quantized(xb, wb, 4, 128)["wq"])
    assert np.array_equal(r48["xq"], o.linear_quantized(xb, wb, 8, 128)["xq"])


def test_static_scale_calibration_is_max_of_dynamic_scales():
    draws = [activations(10, 256, n_outliers=3, outlier_scale=8, seed=s) for s in range(3)]
    s = o.calibrate_static_scale(draws, 4, 64)
    dyn = max(o.act_hadamard_quant(d, 4, 64)[1].max() for d in draws)
    assert s == dyn
    q, sx = o.act_hadamard_quant(draws[0], 4, 64, static_scale=s)
    assert np.all(sx == s) and q.min() >= -7 and q.max() <= 7
