"""ctypes binding of ``libmoe_mxfp4.so``: one Python function per C entry point,
same names, arguments marshalled only (pointers as ints, sizes as ints).

Loading fails loudly when the library has not been built; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_WORKSPACE_TOO_SMALL = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE_TIMEOUT = -5
MOE_ERR_NAN_SCALE = -6

MOE_WEIGHTS_GATEUP = 0
MOE_WEIGHTS_DOWN = 1
MOE_ROUTE_FROM_LOGITS = 1
MOE_ROUTE_GATING_SOFTMAX_ALL = 2
MOE_ROUTE_GATING_SIGMOID = 4
MOE_PEAK_MXF4 = 0
MOE_PEAK_BF16 = 1

# every symbol the header declares, with its C signature
_P = ctypes.c_void_p
_I = ctypes.c_int
_S = ctypes.c_size_t
SIGNATURES = {
    "moe_error_string": (ctypes.c_char_p, [_I]),
    "moe_prepared_weight_bytes": (_S, [_I, _I, _I, _I]),
    "moe_prepare_weights": (_I, [_P, _P, _I, _I, _I, _I, _P, _S, _P]),
    "moe_prepared_weight_bytes_bf16": (_S, [_I, _I, _I, _I]),
    "moe_prepare_weights_bf16": (_I, [_P, _I, _I, _I, _I, _P, _S, _P]),
    "moe_tile_rows": (_I, [_I, _I, _I]),
    "moe_max_tiles": (_I, [_I, _I, _I, _I]),
    "moe_workspace_bytes": (_S, [_I, _I, _I, _I, _I]),
    "moe_route": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _S, _P]),
    "moe_route_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P]),
    "moe_route_noalloc_status": (_I, [ctypes.POINTER(_I), _P]),
    "moe_build_tile_table": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "moe_mxfp4_gateup_swiglu": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P, _S, _P]),
    "moe_mxfp4_down_combine": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _S, _P, _P]),
    "moe_hidden_dequant": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _S, _P, _P]),
    "moe_forward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _S, _P, _P, _P, _P]),
    "moe_forward_gated": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _S, _P, _P, _P, _P]),
    "moe_forward_norm": (_I, [_P, _P, _P, ctypes.c_float, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _S, _P, _P,
                              _P, _P, _P]),
    "moe_forward_bf16": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _S, _P, _P, _P, _P]),
    "moe_forward_timed": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _S, _P, _P, _P, _P, _P]),
    "moe_forward_launches": (_I, [_I, _I, _I, _I, _I]),
    "moe_get_device_status": (_I, [_P, _S, ctypes.POINTER(_I), _P]),
    "moe_tensor_peak": (_I, [_I, _I, ctypes.POINTER(ctypes.c_double), _P]),
    "moe_set_wait_limit_ns": (_I, [ctypes.c_ulonglong]),
}

_lib = None


def load() -> ctypes.CDLL:
    """The loaded library (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with mxfp4_expert_layer_gb300.build.build() "
                               "(the CUDA library is required; there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = load().moe_error_string(status).decode()
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


def check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise MoEError(fn, status)


def _call(name):
    def f(*args):
        return getattr(load(), name)(*args)
    f.__name__ = name
    f.__doc__ = f"Direct call of the C entry point {name} (see include/moe_mxfp4.h)."
    return f


moe_error_string = _call("moe_error_string")
moe_prepared_weight_bytes = _call("moe_prepared_weight_bytes")
moe_prepare_weights = _call("moe_prepare_weights")
moe_prepared_weight_bytes_bf16 = _call("moe_prepared_weight_bytes_bf16")
moe_prepare_weights_bf16 = _call("moe_prepare_weights_bf16")
moe_tile_rows = _call("moe_tile_rows")
moe_max_tiles = _call("moe_max_tiles")
moe_workspace_bytes = _call("moe_workspace_bytes")
moe_route = _call("moe_route")
moe_route_noalloc = _call("moe_route_noalloc")
moe_route_noalloc_status = _call("moe_route_noalloc_status")
moe_build_tile_table = _call("moe_build_tile_table")
moe_mxfp4_gateup_swiglu = _call("moe_mxfp4_gateup_swiglu")
moe_mxfp4_down_combine = _call("moe_mxfp4_down_combine")
moe_hidden_dequant = _call("moe_hidden_dequant")
moe_forward = _call("moe_forward")
moe_forward_gated = _call("moe_forward_gated")
moe_forward_norm = _call("moe_forward_norm")
moe_forward_bf16 = _call("moe_forward_bf16")
moe_forward_timed = _call("moe_forward_timed")
moe_forward_launches = _call("moe_forward_launches")
moe_get_device_status = _call("moe_get_device_status")
moe_tensor_peak = _call("moe_tensor_peak")
moe_set_wait_limit_ns = _call("moe_set_wait_limit_ns")
