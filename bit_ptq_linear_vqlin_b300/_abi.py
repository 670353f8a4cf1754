"""ctypes declarations of libvqlin.so (the C ABI in include/vqlin.h).

Loading fails loudly: there is no fallback implementation of any entry point.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvqlin.so")

STATUS_NAMES = {
    0: "VQLIN_OK",
    1: "VQLIN_ERR_INVALID_ARG",
    2: "VQLIN_ERR_UNSUPPORTED_SHAPE",
    3: "VQLIN_ERR_MISALIGNED",
    4: "VQLIN_ERR_CUDA",
    5: "VQLIN_ERR_TIMEOUT",
    6: "VQLIN_ERR_DEVICE_ASSERT",
}

_p = ctypes.c_void_p
_i = ctypes.c_int

# name -> (restype, argtypes); the order and meaning follow include/vqlin.h
SIGNATURES = {
    "vqlin_version": (_i, []),
    "vqlin_status_string": (ctypes.c_char_p, [_i]),
    "vqlin_last_error_message": (ctypes.c_char_p, []),
    "vqlin_get_last_device_error": (_i, [_p]),
    "vqlin_quantize_weights_rtn": (_i, [_p, _i, _i, _i, _i, _i, _i, _p, _p, _p, _p]),
    "vqlin_act_hadamard_quant": (_i, [_p, _i, _i, _i, _i, _p, _p, _p, _p]),
    "vqlin_linear_w4a4": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _p]),
    "vqlin_linear_w4a4_static": (_i, [_p, _p, _i, _p, _p, _p, _p, _p, _i, _i, _i, _p]),
    "vqlin_linear_w4a4_static_scaled": (_i, [_p, _p, _p, _i, _p, _p, _p, _p, _p, _i, _i, _i, _p]),
    "vqlin_linear_w4a4_static_noalloc": (_i, [_p, _p, _i, _p, _p, _p, _p, _i, _i, _i, _p]),
    "vqlin_linear_w8a8": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _p]),
    "vqlin_linear_w4a8": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _p]),
    "vqlin_debug_gemm_w4a8_s32": (_i, [_p, _p, _p, _i, _i, _i, _p]),
    "vqlin_linear_w4a16": (_i, [_p, _p, _p, _p, _i, _p, _p, _i, _i, _i, _p]),
    "vqlin_linear_bf16_ref": (_i, [_p, _p, _p, _p, _i, _i, _i, _p]),
    "vqlin_debug_gemm_s32": (_i, [_i, _p, _p, _p, _i, _i, _i, _p]),
    "vqlin_debug_gemm_withheld_loads": (_i, [_i, _p, _p, _p, _i, _i, _i, ctypes.c_uint64, _p]),
    "vqlin_debug_w4a16_withheld_loads": (_i, [_p, _p, _p, _p, _i, _p, _i, _i, _i, ctypes.c_uint64, _p]),
    "vqlin_composite_rotation_prepare": (_i, [_p, _i, _i, _i, _p, _p, _p]),
    "vqlin_act_adaln_hadamard_quant": (_i, [_p, _i, _i, _i, _i, _p, _p, ctypes.c_float, _p, _p, _p, _p]),
    "vqlin_kernel_launch_count": (_i, [_p]),
    "vqlin_init": (_i, []),
    "vqlin_shutdown": (_i, []),
    "vqlin_quantize_weights_rtn_scaled": (_i, [_p, _i, _i, _i, _i, _p, _p, _p, _p]),
    "vqlin_act_hadamard_quant_scaled": (_i, [_p, _i, _i, _i, _i, _p, _p, _p, _p, _p]),
    "vqlin_quantize_weights_composite": (_i, [_p, _i, _i, _i, _i, _p, _p, _p, _p, _p]),
    "vqlin_act_composite_quant": (_i, [_p, _i, _i, _i, _i, _p, _p, _p, _p, _p]),
    "vqlin_measure_mma_rate": (_i, [_i, _i, _i, _i, _i, _i, _i, _p, ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_double), _p]),
}

_lib = None


class VqlinError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        name = STATUS_NAMES.get(status, f"status {status}")
        super().__init__(f"{what}: {name}" + (f" ({detail})" if detail else ""))


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libvqlin.so once and declare every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python bit_ptq_linear_vqlin_b300/build.py` "
            "(the library has no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int, what: str) -> None:
    if status != 0:
        detail = load().vqlin_last_error_message().decode("utf-8", "replace")
        raise VqlinError(status, what, detail)
