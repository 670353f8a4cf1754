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
