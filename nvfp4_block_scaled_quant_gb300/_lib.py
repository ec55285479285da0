"""ctypes binding of the C ABI declared in include/nvfp4.h (argument marshalling only).

Loading fails loudly when the shared library is missing: there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import re
import threading
from ctypes import POINTER, Structure, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_uint32, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnvfp4_gb300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "nvfp4.h")

# status codes and flags (mirrors the header)
OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED_SHAPE = 2
ERR_MISALIGNED = 3
ERR_WORKSPACE = 4
ERR_CUDA = 5
ERR_DEVICE_FAULT = 6
ERR_TIMEOUT = 7
ERR_UNSUPPORTED_DEVICE = 8
GS_DYNAMIC = 0
GS_STATIC = 1
SF_SWIZZLED = 0
SF_LINEAR = 1
PREP_PLAIN = 0
PREP_W13_INTERLEAVE = 1
DEVERR_BAD_EXPERT_ID = 1
DEVERR_PIPELINE_TIMEOUT = 2
DEVERR_INTERNAL = 4
LINEAR_NOALLOC_MAX_BYTES = 4 << 20


ABI_VERSION = 6  # NVFP4_ABI_VERSION of the header these signatures follow


class MoeWsLayout(Structure):
    _fields_ = [(n, c_size_t) for n in ("counts", "offsets", "pad_offsets", "tile_offsets", "sorted_idx",
                                         "inv_idx", "dest_rows", "tile_table", "amax_partials", "xq", "xsf", "hq", "hsf", "y_acc", "total")]
    _fields_ += [("rows_capacity", c_int64)]


P = c_void_p
I64 = c_int64
_SIGNATURES = {
    "nvfp4_abi_version": (c_int, []),
    "nvfp4_status_string": (c_char_p, [c_int]),
    "nvfp4_last_error_string": (c_char_p, []),
    "nvfp4_get_device_error": (c_int, [P, POINTER(c_int32)]),
    "nvfp4_sf_bytes": (c_size_t, [I64, I64]),
    "nvfp4_quantize_workspace_bytes": (c_size_t, [I64, I64]),
    "nvfp4_quantize_act": (c_int, [P, I64, I64, I64, c_int, P, P, P, c_int, P, c_size_t, P]),
    "nvfp4_prepare_weights": (c_int, [P, P, I64, I64, I64, c_int, P, P, P]),
    "nvfp4_prepared_weight_bytes": (c_size_t, [I64, I64, I64]),
    "nvfp4_rmsnorm_quantize_workspace_bytes": (c_size_t, [I64, I64]),
    "nvfp4_rmsnorm": (c_int, [P, I64, I64, I64, P, c_float, P, P]),
    "nvfp4_rmsnorm_quantize": (c_int, [P, I64, I64, I64, P, c_float, c_int, P, P, P, c_int, P, P, c_size_t, P]),
    "nvfp4_linear_workspace_bytes": (c_size_t, [I64, I64]),
    "nvfp4_linear": (c_int, [P, I64, I64, I64, P, P, P, c_int, P, P, P, c_size_t, P]),
    "nvfp4_gemm": (c_int, [P, P, P, I64, I64, I64, P, P, P, P, P]),
    "nvfp4_linear_noalloc": (c_int, [P, I64, I64, I64, P, P, P, c_int, P, P, P]),
    "nvfp4_grouped_linear_workspace_bytes": (c_size_t, [I64, I64, I64]),
    "nvfp4_grouped_linear": (c_int, [P, I64, I64, I64, I64, P, P, P, c_int, P, P, P, c_size_t, P]),
    "nvfp4_moe_route": (c_int, [P, I64, c_int, I64, P, P, P, P, P]),
    "nvfp4_router_prepare_workspace_bytes": (c_size_t, [I64, I64]),
    "nvfp4_router_prepare": (c_int, [P, P, P, I64, I64, P, P, c_size_t, P]),
    "nvfp4_router_workspace_bytes": (c_size_t, [I64, I64]),
    "nvfp4_router": (c_int, [P, I64, I64, P, I64, c_int, P, P, P, P, c_size_t, P]),
    "nvfp4_moe_workspace_layout": (c_int, [I64, I64, I64, I64, c_int, c_int, POINTER(MoeWsLayout)]),
    "nvfp4_moe_workspace_bytes": (c_size_t, [I64, I64, I64, I64, c_int, c_int]),
    "nvfp4_moe_forward": (c_int, [P, I64, I64, I64, I64, c_int, P, P, P, P, P, P, P, P, P, P, P, P, P, c_int, P, P,
                                  P, P, c_size_t, P]),
    "nvfp4_moe_dispatch": (c_int, [P, I64, I64, I64, I64, c_int, P, c_int, c_int, P, P, c_size_t, P]),
    "nvfp4_moe_w13": (c_int, [I64, I64, I64, I64, c_int, P, P, P, P, P, P, P, P, P, P, c_size_t, P]),
    "nvfp4_moe_w2": (c_int, [I64, I64, I64, I64, c_int, P, P, P, P, P, P, P, P, P, c_size_t, P]),
    "nvfp4_moe_finalize": (c_int, [I64, I64, I64, I64, c_int, c_int, P, P, c_size_t, P]),
    "nvfp4_debug_wait_timeout": (c_int, [c_uint32, P]),
}

_lib = None
_lock = threading.Lock()


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"nvfp4 status {status}: {detail}")
        self.status = status
        self.detail = detail


def declared_functions() -> list:
    """Names of the functions include/nvfp4.h declares (parsed from the header text)."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"NVFP4_API\s+[\w\s\*]*?\b(nvfp4_\w+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()'); "
                    "this package has no CPU or fallback path")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def check(status: int) -> None:
    if status != OK:
        detail = lib().nvfp4_last_error_string().decode(errors="replace")
        raise Nvfp4Error(status, detail)


def call(name: str, *args) -> None:
    check(getattr(lib(), name)(*args))
