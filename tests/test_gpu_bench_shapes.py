"""Parity at the exact shapes the benchmark times, and the W4A16 bounded waits.

The benchmark's largest launches take plans the smaller parity cases do not
reach (multi-wave grids, the chunked int8 sums, the split-K GEMV at K = 11008),
so each is checked here at its full size:
  * W4A4 / W8A8 / W4A8 projections given identical codes: against the
    oracle's float64 epilogue of the exact integer GEMM, every output within
    one bf16 ulp plus the float32 epilogue's rounding (float(acc) * s_x * s_w
    + bias takes four float32 roundings, each within 2^-24 of the magnitudes
    involved: where the terms cancel, that is many ulps of a small result),
    and fewer than 1% of outputs differing at all;
  * W4A16: relative Frobenius error <= 2e-3 against the oracle, both sides
    rounded to bf16;
  * the W4A16 tensor-core kernel with every load withheld reports a timeout,
    and the next call is correct.
Shapes: the prefix backbone (816 tokens; q|k|v and gate|up fused along N, o
and down at W8A8) and the Llama-2-7B-shaped projections at 1, 64 and 512
tokens (4096 -> 4096, 4096 -> 11008, 11008 -> 4096).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_ptq_linear_vqlin_b300 as vq  # noqa: E402
from oracle import vqlin_oracle as o  # noqa: E402
from synth import activations, random_codes, sub_rng, weights  # noqa: E402

DEV = torch.device("cuda:0")
GUARD = 4096

LLAMA = ((4096, 4096), (11008, 4096), (4096, 11008))
INT_CASES = [("w4a4", 816, 2560, 2048), ("w4a4", 816, 32768, 2048), ("w8a8", 816, 2048, 2048),
             ("w8a8", 816, 2048, 16384)]
INT_CASES += [(v, M, N, K) for M in (1, 64, 512) for N, K in LLAMA for v in ("w8a8", "w4a4", "w4a8")]
W4A16_CASES = [(M, N, K) for M in (1, 4, 64, 512) for N, K in LLAMA]


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def bf16_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def guarded(shape, dtype):
    n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
    raw = torch.full((GUARD + n + GUARD,), 0xA5, dtype=torch.uint8, device=DEV)
    return raw, raw[GUARD:GUARD + n].view(dtype).view(*shape)


def check_guard(raw):
    torch.cuda.synchronize()
    assert bool((raw[:GUARD] == 0xA5).all()), "write before the output buffer"
    assert bool((raw[-GUARD:] == 0xA5).all()), "write after the output buffer"


def encode_act(c, bits):
    if bits == 4:
        return torch.from_numpy(o.encode_act_int4(c)).to(DEV)
    return torch.from_numpy(o.encode_act_int8(c).view(np.int16)).to(DEV)


def pack_codes(c, bits):
    return torch.from_numpy(o.pack_int4(c) if bits == 4 else o.pack_int8(c)).to(DEV)


@pytest.mark.parametrize("case", INT_CASES, ids=lambda c: "%s-%dx%dx%d" % c)
def test_projection_at_bench_shape(case):
    variant, M, N, K = case
    abits, wbits = {"w4a4": (4, 4), "w8a8": (8, 8), "w4a8": (8, 4)}[variant]
    qa, qw = (7 if abits == 4 else 127), (7 if wbits == 4 else 127)
    tags = (variant, M, N, K)
    xq = random_codes((M, K), -qa, qa, seed=61, tags=tags + ("x",))
    wq = random_codes((N, K), -qw, qw, seed=62, tags=tags + ("w",))
    rng = sub_rng(63, *tags)
    sx = rng.uniform(0.01, 0.2, M).astype(np.float32)
    sw = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    bias = weights(1, N, std=0.5, seed=64, tags=tags)[0]
    raw, y = guarded((M, N), torch.bfloat16)
    fn = {"w4a4": vq.linear_w4a4, "w8a8": vq.linear_w8a8, "w4a8": vq.linear_w4a8}[variant]
    fn(encode_act(xq, abits), torch.from_numpy(sx).to(DEV), pack_codes(wq, wbits), torch.from_numpy(sw).to(DEV),
       to_dev_bf16(bias), out=y)
    check_guard(raw)
    vq.get_last_device_error()
    acc = o.int_gemm(xq, wq)
    ref = o.linear_epilogue(acc, sx, sw, bias)
    yb = bf16_bits(y)
    a, r = o.bf16_to_f64(yb), o.bf16_to_f64(ref)
    terms = np.abs(acc.astype(np.float64) * sx.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :])
    terms += np.abs(o.bf16_to_f64(bias))[None, :]
    big = np.maximum(np.abs(a), np.abs(r))
    ulp = np.exp2(np.floor(np.log2(np.maximum(big, 2.0 ** -126))) - 7)
    bound = ulp + 2.0 ** -21 * terms
    excess = np.abs(a - r) / bound
    assert excess.max() <= 1.0, f"worst error {excess.max():.3f} of its bound"
    off = (yb != ref).mean()
    assert off < 0.01, f"{off:.4f} of outputs differ"


@pytest.mark.parametrize("MNK", W4A16_CASES, ids=lambda c: "%dx%dx%d" % c)
def test_w4a16_at_bench_shape(MNK):
    M, N, K = MNK
    Xb = activations(M, K, n_outliers=int(round(0.005 * K)), outlier_scale=50, seed=71, tags=MNK)
    Wb = weights(N, K, seed=72, tags=MNK)
    bias = weights(1, N, std=0.5, seed=73, tags=MNK)[0]
    q, s, z = vq.quantize_weights_rtn(to_dev_bf16(Wb), 4, False, 128, 0)
    raw, y = guarded((M, N), torch.bfloat16)
    vq.linear_w4a16(to_dev_bf16(Xb), q, s, z, 128, to_dev_bf16(bias), out=y)
    check_guard(raw)
    vq.get_last_device_error()
    ref_w = o.quantize_weights_rtn(Wb, 4, False, 128, 0)
    ref = o.linear_w4a16(Xb, ref_w["q"], ref_w["s"], ref_w["z"], 128, bias)
    a, b = o.bf16_to_f64(bf16_bits(y)), o.bf16_to_f64(ref)
    err = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert err <= 2e-3, f"relative Frobenius error {err}"


@pytest.mark.parametrize("MNK", [(50, 256, 1024), (64, 1024, 4096)])
def test_w4a16_bounded_wait_reports_timeout(MNK):
    # the tile producer withholds every load: the expanders', issuers' and
    # drains' waits run out (10 ms), the kernel records a timeout, frees its
    # tensor memory and exits; the context stays usable and the next call is
    # correct
    M, N, K = MNK
    Xb = activations(M, K, seed=81, tags=MNK)
    Wb = weights(N, K, seed=82, tags=MNK)
    X = to_dev_bf16(Xb)
    q, s, z = vq.quantize_weights_rtn(to_dev_bf16(Wb), 4, False, 128, 0)
    vq.get_last_device_error()
    vq.debug_w4a16_withheld_loads(X, q, s, z, 128, limit_ns=10_000_000)
    with pytest.raises(vq.VqlinError, match="TIMEOUT"):
        vq.get_last_device_error()
    vq.get_last_device_error()   # the status word was cleared
    y = vq.linear_w4a16(X, q, s, z, 128)
    vq.get_last_device_error()
    ref_w = o.quantize_weights_rtn(Wb, 4, False, 128, 0)
    ref = o.linear_w4a16(Xb, ref_w["q"], ref_w["s"], ref_w["z"], 128)
    a, b = o.bf16_to_f64(bf16_bits(y)), o.bf16_to_f64(ref)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) <= 2e-3
