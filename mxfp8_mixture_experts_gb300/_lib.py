"""ctypes declarations of libmxmoe.so (the C ABI in include/mxmoe.h).

Loading never falls back to anything: if the library is missing or a symbol
is absent, import fails with an error that says so.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmxmoe.so")

# status codes and enums (mirrors include/mxmoe.h)
MX_OK = 0
MX_ERR_INVALID_ARG = 1
MX_ERR_SHAPE = 2
MX_ERR_ALIGNMENT = 3
MX_ERR_UNSUPPORTED_DEVICE = 4
MX_ERR_CUDA = 5
MX_ERR_DEVICE = 6
MX_ERR_TIMEOUT = 7
MX_ERR_WORKSPACE = 8
MX_ERR_SCRATCH_LIMIT = 9
MX_MODE_ROW, MX_MODE_COL, MX_MODE_BOTH = 1, 2, 3
MX_SCALE_PLAIN, MX_SCALE_SWIZZLED = 0, 1
MX_GEMM_FWD, MX_GEMM_DGRAD, MX_GEMM_WGRAD = 0, 1, 2
MX_OUT_BF16, MX_OUT_F32 = 0, 1
MX_PERMUTE_FP8, MX_PERMUTE_BF16, MX_PERMUTE_BF16_QUANT = 0, 1, 2
MX_ELEM_E4M3, MX_ELEM_E5M2 = 0, 1

_p = C.c_void_p
_i32 = C.c_int32
_i64 = C.c_int64

# name -> (restype, argtypes); every function declared in include/mxmoe.h
SIGNATURES = {
    "mx_status_string": (C.c_char_p, [_i32]),
    "mx_abi_version": (_i32, []),
    "mx_check_device": (_i32, []),
    "mx_selftest_wait_timeout": (_i32, [_i64, _p, _p]),
    "mx_selftest_sigmoid": (_i32, [_p, _i64, _p, _p]),
    "mx_scale_bytes": (_i64, [_i64, _i64, _i32]),
    "mx_quantize": (_i32, [_p, _i64, _i64, _i64, _i32, _i32, _i32, _p, _p, _p, _p, _p]),
    "mx_dequantize": (_i32, [_p, _p, _i64, _i64, _i64, _i32, _i32, _i32, _p, _p]),
    "fp8_quantize_rowmax": (_i32, [_p, _i64, _i64, _p, _p, _p]),
    "moe_route": (_i32, [_p, _i64, _i32, _i32, _p, _p, _p]),
    "moe_rows_cap": (_i64, [_i64, _i32, _i32]),
    "moe_permute_map_workspace_size": (_i64, [_i64, _i32, _i32]),
    "moe_permute_map": (_i32, [_p, _i64, _i32, _i32, _i64, _p, _p, _p, _p, _p, _i64, _p, _p]),
    "moe_permute_map_noalloc": (_i32, [_p, _i64, _i32, _i32, _i64, _p, _p, _p, _p, _p, _p]),
    "moe_permute": (_i32, [_i32, _p, _p, _i64, _i64, _i32, _p, _p, _i64, _p, _p, _i32, _p]),
    "moe_unpermute": (_i32, [_p, _p, _p, _i64, _i64, _i32, _p, _p]),
    "mx_grouped_gemm": (_i32, [_i32, _p, _p, _p, _p, _p, _i32, _i64, _i64, _i64, _p, _i32, _i32, _i32, _p, _p]),
    "mx_wgrad_splitk_workspace_size": (_i64, [_i32, _i64, _i64, _i32]),
    "mx_grouped_gemm_wgrad_splitk": (_i32, [_p, _p, _p, _p, _p, _i32, _i64, _i64, _i64, _i32, _i32, _i32, _p, _i64, _p,
                                            _p, _p]),
    "moe_gemm1_swiglu": (_i32, [_p, _p, _p, _p, _p, _i32, _i64, _i64, _i64, _p, _p, _p, _p, _p]),
    "moe_swiglu_bwd": (_i32, [_p, _p, _i64, _i64, _i32, _p, _p, _p, _p, _p, _p, _p, _p]),
    "moe_gather_quant": (_i32, [_p, _p, _p, _i64, _i64, _i32, _i64, _i32, _i32, _p, _p, _p, _p, _p, _p]),
    "moe_gate_grad": (_i32, [_p, _p, _p, _i64, _i64, _i32, _p, _p]),
    "moe_layer_weights_size": (_i64, [_i64, _i64, _i32]),
    "moe_layer_workspace_size": (_i64, [_i64, _i64, _i64, _i32, _i32]),
    "moe_layer_prep_weights": (_i32, [_p, _p, _i64, _i64, _i32, _p, _i64, _p]),
    "moe_layer_fwd": (_i32, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _i32, _p, _i64, _p, _p, _p]),
    "moe_layer_bwd": (_i32, [_p, _p, _p, _p, _i64, _i64, _i64, _i32, _i32, _i32, _i32, _p, _i64, _p, _p, _p, _p, _p, _p]),
}

_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libmxmoe.so and declare every entry point.  Raises if the library
    has not been built or lacks a declared symbol."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"libmxmoe.so not found at {path}: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)  # AttributeError if missing
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MxError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = load().mx_status_string(code).decode()
        super().__init__(f"{where}: {msg}")


def check(code: int, where: str) -> None:
    if code != MX_OK:
        raise MxError(code, where)
