"""Parity of the composite SVD.Hadamard block rotation (zig-zag permutation,
R_j = V_j H_b / sqrt(b)) with the oracle in oracle/composite_rotation.py.

Bars:
  * the permutation: identical;
  * R_j: within 1e-9 of the oracle's (float64 Jacobi against LAPACK's SVD;
    singular values of Gaussian weights are well separated);
  * weight codes: the rotation is float64 on both sides, rounded once to
    float32, so codes are equal except where the two float64 values fall on
    either side of a float32 rounding point next to a rounding tie (at most
    1e-5 of codes, each off by one); scales within 1e-6;
  * activation codes: the GPU rotates in float32, so codes may differ by one
    only within 1e-4 of a tie of the exact quotient, at most 1e-4 of codes;
    scales within 1e-5;
  * the whole projection through the integer GEMM: relative Frobenius error
    <= 1e-3 against linear_quantized_composite, both sides rounded to bf16.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_ptq_linear_vqlin_b300 as vq  # noqa: E402
from oracle import composite_rotation as cr  # noqa: E402
from oracle import vqlin_oracle as o  # noqa: E402
from synth import activations, weights  # noqa: E402

DEV = torch.device("cuda:0")


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def bf16_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def decode_act(q, bits):
    q = q.cpu().numpy()
    return o.decode_act_int4(q) if bits == 4 else o.decode_act_int8(q.view(np.uint16))


def unpack_w(q, bits):
    q = q.cpu().numpy().view(np.uint8)
    return o.unpack_int4(q, signed=True) if bits == 4 else o.unpack_int8(q)


def _case(M, N, K, seed):
    Xb = activations(M, K, n_outliers=max(1, K // 100), outlier_scale=30, seed=seed, tags=("comp", M, K))
    Wb = weights(N, K, seed=seed + 1, tags=("comp", N, K))
    return Xb, Wb


@pytest.mark.parametrize("b", [64, 128])
@pytest.mark.parametrize("NK", [(512, 1024), (256, 512)])
def test_prepare_matches_oracle(b, NK):
    N, K = NK
    _, Wb = _case(4, N, K, 101)
    perm, R = vq.composite_rotation_prepare(to_dev_bf16(Wb), b)
    vq.get_last_device_error()
    W = o.bf16_to_f64(Wb)
    perm_ref = cr.zigzag_permutation(W, b)
    np.testing.assert_array_equal(perm.cpu().numpy(), perm_ref)
    R_ref = cr.block_rotations(W, perm_ref, b)
    err = np.abs(R.cpu().numpy() - R_ref).max()
    assert err < 1e-9, f"R differs by {err}"
    # each R_j is orthogonal
    Rg = R.cpu().numpy()
    eye = np.eye(b)
    assert max(np.abs(Rg[j] @ Rg[j].T - eye).max() for j in range(K // b)) < 1e-12


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("b", [64, 128])
def test_composite_weight_codes(bits, b):
    N, K = 384, 1024
    _, Wb = _case(4, N, K, 111)
    Wd = to_dev_bf16(Wb)
    perm, R = vq.composite_rotation_prepare(Wd, b)
    q, s = vq.quantize_weights_composite(Wd, bits, b, perm, R)
    vq.get_last_device_error()
    W = o.bf16_to_f64(Wb)
    perm_ref = cr.zigzag_permutation(W, b)
    R_ref = cr.block_rotations(W, perm_ref, b)
    q_ref, s_ref = o.rtn_symmetric_rows(cr.composite_rotate(W, perm_ref, R_ref).astype(np.float32), bits)
    np.testing.assert_allclose(s.cpu().numpy(), s_ref, rtol=1e-6, atol=0)
    diff = unpack_w(q, bits).astype(np.int64) - q_ref.astype(np.int64)
    assert np.abs(diff).max() <= 1
    assert np.count_nonzero(diff) <= max(1, int(1e-5 * diff.size))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("b", [64, 128])
def test_composite_activation_codes(bits, b):
    M, N, K = 77, 256, 2048
    Xb, Wb = _case(M, N, K, 121)
    perm, R = vq.composite_rotation_prepare(to_dev_bf16(Wb), b)
    q, s = vq.act_composite_quant(to_dev_bf16(Xb), bits, b, perm, R)
    vq.get_last_device_error()
    W = o.bf16_to_f64(Wb)
    perm_ref = cr.zigzag_permutation(W, b)
    R_ref = cr.block_rotations(W, perm_ref, b)
    exact = cr.composite_rotate(o.bf16_to_f64(Xb), perm_ref, R_ref)
    q_ref, s_ref = o.rtn_symmetric_rows(exact.astype(np.float32), bits)
    np.testing.assert_allclose(s.cpu().numpy(), s_ref, rtol=1e-5, atol=0)
    diff = decode_act(q, bits).astype(np.int64) - q_ref.astype(np.int64)
    bad = np.nonzero(diff)
    assert np.all(np.abs(diff) <= 1)
    quot = exact / np.where(s_ref > 0, s_ref, 1).astype(np.float64)[:, None]
    frac = np.abs(quot[bad] - np.floor(quot[bad]) - 0.5)
    assert np.all(frac < 1e-4), "a code differs away from a rounding tie"
    assert bad[0].size <= 1e-4 * diff.size


@pytest.mark.parametrize("bits,act_bits", [(4, 4), (8, 8), (4, 8)], ids=["w4a4", "w8a8", "w4a8"])
@pytest.mark.parametrize("b", [64, 128])
def test_linear_quantized_composite(bits, act_bits, b):
    M, N, K = 50, 640, 1024
    Xb, Wb = _case(M, N, K, 131)
    bias = weights(1, N, std=0.5, seed=133)[0]
    Wd, Xd = to_dev_bf16(Wb), to_dev_bf16(Xb)
    perm, R = vq.composite_rotation_prepare(Wd, b)
    wq, sw = vq.quantize_weights_composite(Wd, bits, b, perm, R)
    xq, sx = vq.act_composite_quant(Xd, act_bits, b, perm, R)
    fn = {(4, 4): vq.linear_w4a4, (8, 8): vq.linear_w8a8, (4, 8): vq.linear_w4a8}[(bits, act_bits)]
    y = fn(xq, sx, wq, sw, to_dev_bf16(bias))
    vq.get_last_device_error()
    ref = cr.linear_quantized_composite(Xb, Wb, bits, b, bias_bits=bias, act_bits=act_bits)
    a, r = o.bf16_to_f64(bf16_bits(y)), o.bf16_to_f64(ref["y"])
    err = np.linalg.norm(a - r) / np.linalg.norm(r)
    assert err <= 1e-3, f"relative Frobenius error {err}"


def test_composite_rejects_bad_arguments():
    X = torch.zeros((4, 96), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(vq.VqlinError):
        vq.composite_rotation_prepare(X, 64)          # K % b
    X = torch.zeros((4, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(vq.VqlinError):
        vq.composite_rotation_prepare(X, 32)          # block size
