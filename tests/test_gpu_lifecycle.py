"""vqlin_init / vqlin_shutdown: the library's per-device state (status word,
cuBLASLt handle and workspace of the bf16 baseline) made ahead of use,
released, and made again on the next call."""
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


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def test_init_shutdown_cycle():
    Xb, Wb = activations(8, 256, seed=301), weights(64, 256, seed=302)
    ref = o.bf16_to_f64(o.linear_bf16(Xb, Wb))
    for _ in range(2):
        vq.init()
        vq.init()   # idempotent
        y = vq.linear_bf16_ref(to_dev_bf16(Xb), to_dev_bf16(Wb))
        a = o.bf16_to_f64(y.cpu().view(torch.int16).numpy().view(np.uint16))
        assert np.linalg.norm(a - ref) / np.linalg.norm(ref) <= 1e-3
        vq.shutdown()
        vq.shutdown()   # nothing left: a no-op
    # first use after shutdown creates the state again
    y = vq.linear_bf16_ref(to_dev_bf16(Xb), to_dev_bf16(Wb))
    vq.get_last_device_error()
    a = o.bf16_to_f64(y.cpu().view(torch.int16).numpy().view(np.uint16))
    assert np.linalg.norm(a - ref) / np.linalg.norm(ref) <= 1e-3


def test_launch_count_matches_the_kernels_of_each_call():
    # the count the bench reports as gpu_launches: one kernel per call, two for
    # the static-scale projection at 32 k-blocks or more (activation kernel +
    # codes GEMM), none for the cuBLAS baseline
    def launches(fn):
        n0 = vq.kernel_launch_count()
        fn()
        torch.cuda.synchronize()
        return vq.kernel_launch_count() - n0

    M = 50
    for K, expect in ((1024, 1), (4096, 2)):
        X, W = to_dev_bf16(activations(M, K, seed=311)), to_dev_bf16(weights(256, K, seed=312))
        wq, sw = vq.quantize_weights_rtn(W, 4, True, 0, 128)
        st = torch.tensor([0.5], dtype=torch.float32, device=DEV)
        assert launches(lambda: vq.linear_w4a4_static(X, st, wq, sw, 128)) == expect
        assert launches(lambda: vq.act_hadamard_quant(X, 4, 128)) == 1
        q16, s16, z16 = vq.quantize_weights_rtn(W, 4, False, 128, 0)
        assert launches(lambda: vq.linear_w4a16(X, q16, s16, z16, 128)) == 1
        assert launches(lambda: vq.linear_bf16_ref(X, W)) == 0
    vq.get_last_device_error()
