"""ctypes loader for libkvc.so (the C ABI of include/kvc.h).

No fallback: if the library is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvc.so")

KVC_F32, KVC_BF16, KVC_FP8_E4M3 = 0, 1, 2
STATUS_NAMES = {
    0: "KVC_OK",
    1: "KVC_ERR_ARG",
    2: "KVC_ERR_SHAPE",
    3: "KVC_ERR_OVERFLOW",
    4: "KVC_ERR_LAYER_MISMATCH",
    5: "KVC_ERR_CUDA",
    6: "KVC_ERR_DEVICE_TIMEOUT",
    7: "KVC_ERR_WORKSPACE",
}
KVC_MAX_BATCH = 1024

# (name, restype, argtypes) for every entry point declared in include/kvc.h
_VP, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)
SIGNATURES = [
    ("kvc_create", _I, [ctypes.POINTER(_VP), _I, _I, _I, _I, _I, _I, ctypes.POINTER(_VP), ctypes.POINTER(_VP)]),
    ("kvc_create_paged", _I, [ctypes.POINTER(_VP), _I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_VP),
                              ctypes.POINTER(_VP), _VP]),
    ("kvc_destroy", None, [_VP]),
    ("kvc_set_kv_scales", _I, [_VP, _I, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]),
    ("kvc_append", _I, [_VP, _I, _VP, _VP, _I, _I32P, _VP]),
    ("kvc_workspace_bytes", _SZ, [_VP, _I, _I]),
    ("kvc_gqa_attention", _I, [_VP, _I, _VP, _I, _I, _I32P, _VP, _VP, _SZ, _VP]),
    ("kvc_append_attention", _I, [_VP, _I, _VP, _VP, _VP, _I, _I, _I32P, _VP, _VP, _SZ, _VP]),
    ("kvc_gqa_attention_tree", _I, [_VP, _I, _VP, _I, _I, _I32P, _I32P, _VP, _VP, _SZ, _VP]),
    ("kvc_append_attention_tree", _I, [_VP, _I, _VP, _VP, _VP, _I, _I, _I32P, _I32P, _VP, _VP, _SZ, _VP]),
    ("kvc_append_attention_host", _I, [_VP, _I, _VP, _VP, _VP, _I, _I, _I32P, _VP, _VP, _SZ, _VP]),
    ("kvc_host_copies_done", _I, [_VP, _VP]),
    ("kvc_gqa_attention_noalloc", _I, [_VP, _I, _VP, _I, _I, _I32P, _VP, _VP]),
    ("kvc_noalloc_status", _I, [_VP, _I32P]),
    ("kvc_set_window", _I, [_VP, _I, _I]),
    ("kvc_truncate", _I, [_VP, _I64P]),
    ("kvc_reset", _I, [_VP]),
    ("kvc_set_lens", _I, [_VP, _I, _I64P]),
    ("kvc_get_lens", _I, [_VP, _I, _I64P]),
    ("kvc_length", _I, [_VP, _I64P]),
    ("kvc_device_status", _I, [_VP, _VP, _VP, _I32P]),
    ("kvc_selftest_bounded_wait", _I, [_VP, ctypes.c_uint64, _VP]),
    ("kvc_device_lens_bytes", _SZ, [_VP]),
    ("kvc_lens_to_device", _I, [_VP, _VP, _VP]),
    ("kvc_lens_from_device", _I, [_VP, _VP]),
    ("kvc_decode_step", _I, [_VP, _I, _VP, _VP, _VP, _I, _I, _VP, _VP, _VP, _SZ, _VP]),
    ("kvc_kernel_launches", ctypes.c_uint64, [_VP]),
    ("kvc_last_error", ctypes.c_char_p, []),
    ("kvc_version", ctypes.c_char_p, []),
]

_lib = None


class KVCError(ValueError):
    """A kvc_* call returned a non-zero status."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


def lib() -> ctypes.CDLL:
    """The loaded library; raises RuntimeError if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libkvc.so not found at {LIB_PATH}; build it with "
                "`python -m gqa_attention_preallocated_gb300.build` (there is no CPU fallback)"
            )
        handle = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def check(status: int) -> None:
    if status != 0:
        raise KVCError(status, lib().kvc_last_error().decode())
