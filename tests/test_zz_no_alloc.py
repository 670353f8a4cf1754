"""The W4A4 static-scale projection for callers that cannot allocate device
memory (vqlin_linear_w4a4_static_noalloc): no code buffer of the caller's, the
library's fixed device array instead.

Called through the C ABI (ctypes), twice in a row with different inputs, each
output checked against vqlin_linear_w4a4_static (caller's buffer) within the
W4A4 tolerance of the parity tests.  The file sorts last, so a run that stops at
the first failure has already run every other test; it also passes alone in a
fresh process (the first call sets the array up).
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU machines too
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bit_ptq_linear_vqlin_b300 as vq  # noqa: E402
from oracle import vqlin_oracle as o  # noqa: E402
from synth import activations, weights  # noqa: E402

DEV = torch.device("cuda:0")


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _rel_fro(a_bits, b_bits):
    a, b = o.bf16_to_f64(a_bits), o.bf16_to_f64(b_bits)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _case(M, N, K, hb, seed):
    Xb = activations(M, K, n_outliers=max(1, K // 200), outlier_scale=20, seed=seed)
    Wb = weights(N, K, seed=seed + 1)
    bias = _dev_bf16(weights(1, N, std=0.5, seed=seed + 2)[0])
    s = o.calibrate_static_scale([activations(M, K, n_outliers=max(1, K // 200), outlier_scale=20, seed=seed + 3)],
                                 4, hb)
    wq, sw = vq.quantize_weights_rtn(_dev_bf16(Wb), 4, True, 0, hb)
    return _dev_bf16(Xb), torch.tensor([s], dtype=torch.float32, device=DEV), wq, sw, bias


@pytest.mark.parametrize("MNK", [(50, 1024, 1024), (50, 1024, 4096), (16, 384, 20480)])
def test_noalloc_matches_the_buffered_projection_twice(MNK):
    M, N, K = MNK
    hb = 128
    lib = vq._lib
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, seed in enumerate((81, 91)):  # two calls in a row, different inputs
        X, st, wq, sw, bias = _case(M, N, K, hb, seed)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        status = lib.vqlin_linear_w4a4_static_noalloc(_ptr(X), _ptr(st), hb, _ptr(wq), _ptr(sw), _ptr(bias),
                                                      _ptr(y), M, N, K, stream)
        assert status == 0, lib.vqlin_last_error_message().decode()
        ref = vq.linear_w4a4_static(X, st, wq, sw, hb, bias)
        vq.get_last_device_error()
        err = _rel_fro(_bits(y), _bits(ref))
        assert err <= 1e-3, f"call {call}: relative error {err} against vqlin_linear_w4a4_static"


def test_noalloc_rejects_sizes_beyond_its_array():
    lib = vq._lib
    a = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    # 64 x 32768 codes = 2 MiB > the 1 MiB array
    assert lib.vqlin_linear_w4a4_static_noalloc(a, a, 128, a, a, None, a, 64, 128, 32768, None) == 2
    assert b"exceed" in lib.vqlin_last_error_message()
