"""ctypes view of the libbsa C ABI (include/bsa.h).

Argument marshalling only: every step of the hot path runs in libbsa's CUDA
kernels.  Loading fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbsa.so")

SELECT_TOKEN_MAX = 1   # bsa_select_params.flags: per-token query aggregation

STATUS = {
    0: "BSA_OK", 1: "BSA_ERR_INVALID_ARG", 2: "BSA_ERR_SHAPE", 3: "BSA_ERR_UNSUPPORTED",
    4: "BSA_ERR_WORKSPACE", 5: "BSA_ERR_CUDA", 6: "BSA_ERR_DEVICE_TIMEOUT",
}

# Every function declared in include/bsa.h, with its ctypes signature.
_P = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)


class Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seq", ctypes.c_int32), ("hq", ctypes.c_int32),
                ("hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("block", ctypes.c_int32)]


class SelectParams(ctypes.Structure):
    _fields_ = [("centroid_keep", ctypes.c_float), ("rescue_keep", ctypes.c_float),
                ("flags", ctypes.c_int32)]


class VarlenShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("max_seqlen", ctypes.c_int32), ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block", ctypes.c_int32)]


_SP = ctypes.POINTER(Shape)
_VP = ctypes.POINTER(VarlenShape)
_PP = ctypes.POINTER(SelectParams)

SIGNATURES = {
    "bsa_block_meta": (ctypes.c_int, [_SP, _P, _P, _P, _P, _P, _P, _P]),
    "bsa_select_workspace_bytes": (ctypes.c_size_t, [_SP]),
    "bsa_select_mask": (ctypes.c_int, [_SP, _PP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                       _P, _P]),
    "bsa_select_mask_noalloc": (ctypes.c_int, [_SP, _PP, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "bsa_mask_build_workspace_bytes": (ctypes.c_size_t, [_SP]),
    "bsa_mask_build": (ctypes.c_int, [_SP, _PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                      _P, _P]),
    "bsa_prefill_fwd": (ctypes.c_int, [_SP, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P]),
    "bsa_prefill_dense_fwd": (ctypes.c_int, [_SP, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P]),
    "bsa_prefill_layer_workspace_bytes": (ctypes.c_size_t, [_SP]),
    "bsa_prefill_layer": (ctypes.c_int, [_SP, _PP, _P, _P, _P, ctypes.c_float, _P, _P, _P,
                                         ctypes.c_size_t, _P, _P]),
    "bsa_prefill_layer_views": (ctypes.c_int, [_SP, ctypes.POINTER(ctypes.c_size_t)]),
    "bsa_block_meta_fp8": (ctypes.c_int, [_SP, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P]),
    "bsa_select_mask_fp8": (ctypes.c_int, [_SP, _PP, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P, _P,
                                           ctypes.c_size_t, _P, _P]),
    "bsa_prefill_fp8_workspace_bytes": (ctypes.c_size_t, [_SP]),
    "bsa_prefill_fwd_fp8": (ctypes.c_int, [_SP, _P, _P, _P, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_float, _P, _P, ctypes.c_float, _P, _P, _P,
                                           ctypes.c_size_t, _P, _P]),
    "bsa_prefill_dense_fwd_fp8": (ctypes.c_int, [_SP, _P, _P, _P, ctypes.c_float, ctypes.c_float,
                                                 ctypes.c_float, ctypes.c_float, _P, _P, _P,
                                                 ctypes.c_size_t, _P, _P]),
    "bsa_varlen_block_stride": (ctypes.c_int32, [_VP]),
    "bsa_varlen_block_meta": (ctypes.c_int, [_VP, _P, _P, _P, _P, _P, _P, _P, _P]),
    "bsa_varlen_select_workspace_bytes": (ctypes.c_size_t, [_VP]),
    "bsa_varlen_select_mask": (ctypes.c_int, [_VP, _PP, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                              ctypes.c_size_t, _P, _P]),
    "bsa_varlen_prefill_fwd": (ctypes.c_int, [_VP, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                              _P, _P]),
    "bsa_varlen_prefill_dense_fwd": (ctypes.c_int, [_VP, _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                                    _P, _P]),
    "bsa_decode_workspace_bytes": (ctypes.c_size_t, [_VP]),
    "bsa_decode_select": (ctypes.c_int, [_VP, _PP, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                         _P, _P]),
    "bsa_decode_fwd": (ctypes.c_int, [_VP, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P,
                                      ctypes.c_size_t, _P, _P]),
    "bsa_decode_step": (ctypes.c_int, [_VP, _PP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                       _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "bsa_selftest_wait_timeout": (ctypes.c_int, [_P, ctypes.c_uint64, ctypes.c_int32, _P]),
    "bsa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "bsa_version": (ctypes.c_int32, []),
}

_lib = None


class BsaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libbsa.so (once).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"libbsa.so not found at {path}; build it with "
            "`python -m block_sparse_long_kv_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(fn: str, code: int) -> None:
    if code != 0:
        raise BsaError(fn, code)
