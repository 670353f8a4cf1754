"""The AdaLayerNorm fused into the activation kernel
(vqlin_act_adaln_hadamard_quant) against oracle/norm_fusion.py.

Bars: scales within 1e-5 (the GPU's mean, variance and reciprocal root are
float32); codes equal except within 1e-4 of a rounding tie of the exact
quotient, at most 1e-4 of codes; the projection through the W4A4 / W8A8 GEMM
within relative Frobenius error 1e-3 of the oracle's, both rounded to bf16.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_ptq_linear_vqlin_b300 as vq  # noqa: E402
from oracle import norm_fusion as nf  # noqa: E402
from oracle import vqlin_oracle as o  # noqa: E402
from synth import activations, sub_rng, weights  # noqa: E402

DEV = torch.device("cuda:0")
EPS = 1e-6


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def bf16_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def decode_act(q, bits):
    q = q.cpu().numpy()
    return o.decode_act_int4(q) if bits == 4 else o.decode_act_int8(q.view(np.uint16))


def modulation(K, seed):
    rng = sub_rng(seed, "adaln", K)
    return rng.normal(0.0, 0.3, K).astype(np.float32), rng.normal(0.0, 0.5, K).astype(np.float32)


CASES = [(50, 1024, 4, 128), (16, 2048, 4, 64), (7, 4096, 8, 128), (33, 512, 8, 0), (3, 16384, 4, 128),
         (2, 20480, 8, 128), (129, 1024, 4, 128)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "M%d-K%d-b%d-hb%d" % c)
def test_adaln_codes(case):
    M, K, bits, hb = case
    Xb = activations(M, K, n_outliers=max(1, K // 100), outlier_scale=30, seed=401, tags=case)
    sc, sh = modulation(K, 402)
    q, s = vq.act_adaln_hadamard_quant(to_dev_bf16(Xb), bits, hb, torch.from_numpy(sc).to(DEV),
                                       torch.from_numpy(sh).to(DEV), EPS)
    vq.get_last_device_error()
    q_ref, s_ref = nf.adaln_hadamard_quant(Xb, sc.astype(np.float64), sh.astype(np.float64), EPS, bits, hb)
    np.testing.assert_allclose(s.cpu().numpy(), s_ref, rtol=1e-5, atol=0)
    diff = decode_act(q, bits).astype(np.int64) - q_ref.astype(np.int64)
    bad = np.nonzero(diff)
    assert np.all(np.abs(diff) <= 1)
    exact = nf.adaln_rotated_f64(Xb, sc.astype(np.float64), sh.astype(np.float64), EPS, hb)
    quot = exact / np.where(s_ref > 0, s_ref, 1).astype(np.float64)[:, None]
    assert np.all(np.abs(quot[bad] - np.floor(quot[bad]) - 0.5) < 1e-4), "a code differs away from a tie"
    assert bad[0].size <= 1e-4 * diff.size


def test_adaln_static_scale():
    M, K, bits, hb = 50, 1024, 4, 128
    Xb = activations(M, K, n_outliers=10, outlier_scale=30, seed=411)
    sc, sh = modulation(K, 412)
    st = np.float32(0.35)
    q, s = vq.act_adaln_hadamard_quant(to_dev_bf16(Xb), bits, hb, torch.from_numpy(sc).to(DEV),
                                       torch.from_numpy(sh).to(DEV), EPS,
                                       static_scale=torch.tensor([st], dtype=torch.float32, device=DEV))
    vq.get_last_device_error()
    q_ref, s_ref = nf.adaln_hadamard_quant(Xb, sc.astype(np.float64), sh.astype(np.float64), EPS, bits, hb,
                                           static_scale=st)
    np.testing.assert_array_equal(s.cpu().numpy(), s_ref)
    diff = decode_act(q, bits).astype(np.int64) - q_ref.astype(np.int64)
    assert np.abs(diff).max() <= 1 and np.count_nonzero(diff) <= 1e-4 * diff.size


@pytest.mark.parametrize("bits", [4, 8])
def test_adaln_projection(bits):
    M, N, K, hb = 50, 640, 1024, 128
    Xb = activations(M, K, n_outliers=10, outlier_scale=30, seed=421)
    Wb = weights(N, K, seed=422)
    sc, sh = modulation(K, 423)
    wq, sw = vq.quantize_weights_rtn(to_dev_bf16(Wb), bits, True, 0, hb)
    xq, sx = vq.act_adaln_hadamard_quant(to_dev_bf16(Xb), bits, hb, torch.from_numpy(sc).to(DEV),
                                         torch.from_numpy(sh).to(DEV), EPS)
    y = (vq.linear_w4a4 if bits == 4 else vq.linear_w8a8)(xq, sx, wq, sw)
    vq.get_last_device_error()
    wt = o.quantize_weights_rtn(Wb, bits, True, 0, hb)
    q_ref, s_ref = nf.adaln_hadamard_quant(Xb, sc.astype(np.float64), sh.astype(np.float64), EPS, bits, hb)
    ref = o.linear_epilogue(o.int_gemm(q_ref, wt["q"]), s_ref, wt["s"])
    a, r = o.bf16_to_f64(bf16_bits(y)), o.bf16_to_f64(ref)
    assert np.linalg.norm(a - r) / np.linalg.norm(r) <= 1e-3
