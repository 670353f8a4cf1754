"""The C-ABI library loads, exports what include/vqlin.h declares, and
rejects bad arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

from bit_ptq_linear_vqlin_b300 import _abi

HEADER = os.path.join(ROOT, "include", "vqlin.h")
OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3
A = 0x10000  # a 16-byte-aligned address that is never dereferenced: every call
             # below fails a host-side check before anything is launched


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vqlin_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return _abi.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name
        assert name in _abi.SIGNATURES, f"{name} has no ctypes signature"


def test_status_strings(lib):
    for code, name in _abi.STATUS_NAMES.items():
        assert lib.vqlin_status_string(code).decode() == name
    assert lib.vqlin_version() >= 100


def test_act_quant_rejects_bad_arguments(lib):
    f = lib.vqlin_act_hadamard_quant
    assert f(A, 4, 256, 5, 64, None, A, A, None) == INVALID          # bits
    assert f(A, 4, 256, 4, 32, None, A, A, None) == INVALID          # block size
    assert f(A, 4, 96, 4, 64, None, A, A, None) == UNSUPPORTED       # K % b
    assert f(A, 4, 100, 4, 0, None, A, A, None) == UNSUPPORTED       # K % 32
    assert f(A, 4, 1 << 17, 4, 0, None, A, A, None) == UNSUPPORTED   # K too large
    assert f(None, 4, 256, 4, 64, None, A, A, None) == INVALID       # null X
    assert f(A + 8, 4, 256, 4, 64, None, A, A, None) == MISALIGNED   # X
    assert f(A, 4, 256, 4, 64, None, A + 4, A, None) == MISALIGNED   # codes
    assert f(A, -1, 256, 4, 64, None, A, A, None) == INVALID         # M
    assert f(None, 0, 256, 4, 64, None, None, None, None) == OK      # empty: no-op
    assert b"bits" in lib.vqlin_last_error_message() or True


def test_weight_quant_rejects_bad_arguments(lib):
    f = lib.vqlin_quantize_weights_rtn
    assert f(A, 8, 256, 4, 1, 128, 0, A, A, None, None) == INVALID      # sym with groups
    assert f(A, 8, 256, 4, 1, 0, 0, A, A, A, None) == INVALID           # sym with zeros
    assert f(A, 8, 256, 8, 0, 128, 0, A, A, A, None) == INVALID         # asym int8
    assert f(A, 8, 256, 4, 0, 128, 64, A, A, A, None) == INVALID        # asym rotated
    assert f(A, 8, 256, 4, 0, 96, 0, A, A, A, None) == INVALID          # group size
    assert f(A, 8, 320, 4, 0, 128, 0, A, A, A, None) == UNSUPPORTED     # K % group
    assert f(A, 8, 320, 4, 1, 0, 128, A, A, None, None) == UNSUPPORTED  # K % b
    assert f(A, 8, 65536, 4, 1, 0, 0, A, A, None, None) == UNSUPPORTED  # K too large
    assert f(A, 8, 256, 4, 0, 128, 0, A, A, None, None) == INVALID      # null zeros
    assert f(A, 8, 256, 4, 1, 0, 0, A + 2, A, None, None) == MISALIGNED


def test_shutdown_without_state_is_a_no_op(lib):
    # nothing was created on this host (no device): there is nothing to release
    assert lib.vqlin_shutdown() == OK


def test_launch_count_is_host_side(lib):
    # the tally needs no device; rejected calls (no device, bad arguments) launch nothing
    import ctypes
    n = ctypes.c_ulonglong(12345)
    assert lib.vqlin_kernel_launch_count(ctypes.byref(n)) == OK
    before = n.value
    assert lib.vqlin_linear_w4a4(A, A, A, A, None, A, 16, 16, 192, None) == UNSUPPORTED
    assert lib.vqlin_kernel_launch_count(ctypes.byref(n)) == OK and n.value == before
    assert lib.vqlin_kernel_launch_count(None) == INVALID


def test_static_scaled_rejects_bad_arguments(lib):
    f = lib.vqlin_linear_w4a4_static_scaled
    assert f(A, A, None, 128, A, A, None, A, A, 16, 256, 256, None) == INVALID      # null channel scale
    assert f(A, A, A + 4, 128, A, A, None, A, A, 16, 256, 256, None) == MISALIGNED
    assert f(A, A, A, 96, A, A, None, A, A, 16, 256, 256, None) == INVALID          # Hadamard block
    assert f(A, A, A, 128, A, A, None, A, A, 16, 256, 192, None) == UNSUPPORTED     # K % 128
    assert f(A, A, None, 128, A, A, None, A, A, 0, 256, 256, None) == OK            # empty: no-op


def test_linear_rejects_bad_arguments(lib):
    assert lib.vqlin_linear_w4a4(A, A, A, A, None, A, 16, 16, 192, None) == UNSUPPORTED
    assert lib.vqlin_linear_w8a8(A, A, A, A, None, A, 16, 16, 96, None) == UNSUPPORTED
    assert lib.vqlin_linear_w4a4(A, None, A, A, None, A, 16, 16, 256, None) == INVALID
    assert lib.vqlin_linear_w4a4(A + 1, A, A, A, None, A, 16, 16, 256, None) == MISALIGNED
    assert lib.vqlin_linear_w4a4(A, A, A, A, None, A, 0, 16, 256, None) == OK
    assert lib.vqlin_linear_w4a8(A, A, A, A, None, A, 16, 16, 96, None) == UNSUPPORTED       # K % 64
    assert lib.vqlin_linear_w4a8(A, None, A, A, None, A, 16, 16, 128, None) == INVALID       # null sx
    assert lib.vqlin_linear_w4a8(A + 2, A, A, A, None, A, 16, 16, 128, None) == MISALIGNED
    assert lib.vqlin_debug_gemm_w4a8_s32(A, A, None, 16, 16, 128, None) == INVALID          # null acc
    f = lib.vqlin_linear_w4a4_static
    assert f(A, A, 128, A, A, None, A, A, 16, 16, 192, None) == UNSUPPORTED    # K % 128
    assert f(A, A, 32, A, A, None, A, A, 16, 16, 256, None) == INVALID         # block size
    assert f(A, None, 128, A, A, None, A, A, 16, 16, 256, None) == INVALID     # null scale
    assert f(A, A, 128, A, A, None, A, None, 16, 16, 256, None) == INVALID     # null code buffer
    assert f(A + 2, A, 128, A, A, None, A, A, 16, 16, 256, None) == MISALIGNED
    assert f(A, A, 128, A, A, None, A, A + 8, 16, 16, 256, None) == MISALIGNED  # code buffer
    assert f(A, A, 128, A, A, None, A, A, 0, 16, 256, None) == OK              # empty: no-op
    assert lib.vqlin_linear_w4a16(A, A, A, A, 96, None, A, 4, 16, 256, None) == INVALID
    assert lib.vqlin_linear_w4a16(A, A, A, A, 128, None, A, 4, 16, 192, None) == UNSUPPORTED
    assert lib.vqlin_linear_w4a16(A, A, A, None, 128, None, A, 4, 16, 256, None) == INVALID
    assert lib.vqlin_linear_bf16_ref(A, A, None, A, 4, 12, 256, None) == UNSUPPORTED
    assert lib.vqlin_debug_gemm_s32(5, A, A, A, 4, 4, 256, None) == INVALID
    assert lib.vqlin_debug_gemm_s32(4, A, A, None, 4, 4, 256, None) == INVALID
    f = lib.vqlin_act_adaln_hadamard_quant
    assert f(A, 16, 256, 4, 128, None, A, 1e-6, None, A, A, None) == INVALID      # null scale vector
    assert f(A, 16, 256, 4, 128, A, A, -1.0, None, A, A, None) == INVALID         # eps < 0
    assert f(A, 16, 192, 4, 128, A, A, 1e-6, None, A, A, None) == UNSUPPORTED     # K % b
    assert f(A, 16, 256, 4, 128, A + 4, A, 1e-6, None, A, A, None) == MISALIGNED
    assert f(A, 0, 256, 8, 64, A, A, 1e-6, None, A, A, None) == OK               # empty: no-op
    f = lib.vqlin_composite_rotation_prepare
    assert f(A, 16, 256, 32, A, A, None) == INVALID          # block size
    assert f(A, 16, 192, 128, A, A, None) == UNSUPPORTED     # K % b
    assert f(A, 0, 256, 64, A, A, None) == INVALID           # no weights to take the rotation from
    assert f(A, 16, 256, 64, None, A, None) == INVALID       # null perm
    f = lib.vqlin_quantize_weights_composite
    assert f(A, 16, 256, 5, 64, A, A, A, A, None) == INVALID    # bits
    assert f(A, 16, 256, 4, 64, A, None, A, A, None) == INVALID  # null R
    assert f(A, 0, 256, 4, 64, A, A, A, A, None) == OK         # empty: no-op
    f = lib.vqlin_act_composite_quant
    assert f(A, 16, 320, 4, 128, A, A, A, A, None) == UNSUPPORTED   # K % b
    assert f(A + 2, 16, 256, 8, 128, A, A, A, A, None) == MISALIGNED
    assert f(A, 0, 256, 8, 128, A, A, A, A, None) == OK
    f = lib.vqlin_debug_w4a16_withheld_loads
    assert f(A, A, A, A, 128, A, 4, 16, 256, 1000000, None) == INVALID        # M <= 4: the GEMV, no hook
    assert f(A, A, A, A, 128, A, 16, 16, 256, 0, None) == INVALID            # limit 0
    assert f(A, A, A, None, 128, A, 16, 16, 256, 1000000, None) == INVALID   # null zero points
    assert f(A, A, A, A, 128, A, 16, 16, 192, 1000000, None) == UNSUPPORTED  # K % 128
