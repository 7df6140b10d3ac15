"""ctypes declarations for libtq.so (include/tq.h).  Marshalling only."""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtq.so")

TQ_OK = 0
TQ_EINVAL = -1
TQ_EUNSUPPORTED = -2
TQ_EALIGN = -3
TQ_ECUDA = -4
TQ_ENOMEM = -5
TQ_EWORKSPACE = -6
TQ_MSE, TQ_PROD = 0, 1
TQ_BF16, TQ_F32 = 0, 1
TQ_ROT_QR, TQ_ROT_HADAMARD = 0, 1
TQ_STATUS_APPEND_FULL = 200
TQ_STATUS_BAD_CHANNEL = 201

ERROR_NAMES = {TQ_EINVAL: "TQ_EINVAL", TQ_EUNSUPPORTED: "TQ_EUNSUPPORTED", TQ_EALIGN: "TQ_EALIGN",
               TQ_ECUDA: "TQ_ECUDA", TQ_ENOMEM: "TQ_ENOMEM", TQ_EWORKSPACE: "TQ_EWORKSPACE"}

# Every symbol include/tq.h declares, for the export check.
EXPORTED = ["tq_init", "tq_init_ex", "tq_destroy", "tq_row_bytes", "tq_build_params_host",
            "tq_build_params_host_ex", "tq_get_params",
            "tq_quantize", "tq_quantize_kv", "tq_dequantize", "tq_decode_workspace_bytes", "tq_decode_attention",
            "tq_decode_attention_noalloc", "tq_decode_append_attention", "tq_select_outlier_channels",
            "tq_mixed_quantize_scratch_bytes", "tq_mixed_quantize", "tq_mixed_quantize_kv", "tq_mixed_dequantize", "tq_mixed_decode_workspace_bytes",
            "tq_mixed_decode_attention", "tq_device_status", "tq_check_wait_timeout", "tq_last_error"]
NOALLOC_WORKSPACE_BYTES = 4 << 20


class Planes(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("signs", ctypes.c_void_p),
                ("norm", ctypes.c_void_p), ("rnorm", ctypes.c_void_p)]


class TQError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load libtq.so; raises ImportError when the CUDA library has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtq.so not built ({LIB_PATH}); run `python -m kv_cache_vector_18_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    dp = ctypes.POINTER(ctypes.c_double)
    L.tq_init.argtypes = [i32, i32, i32, u64, ctypes.POINTER(vp)]
    L.tq_init_ex.argtypes = [i32, i32, i32, i32, u64, ctypes.POINTER(vp)]
    L.tq_destroy.argtypes = [vp]
    L.tq_row_bytes.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.tq_build_params_host.argtypes = [i32, i32, i32, u64, dp, dp, dp, dp]
    L.tq_build_params_host_ex.argtypes = [i32, i32, i32, i32, u64, dp, dp, dp, dp]
    L.tq_get_params.argtypes = [vp, dp, dp, dp, dp]
    L.tq_quantize.argtypes = [vp, vp, i32, i64, i64, Planes, vp]
    L.tq_quantize_kv.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, Planes, Planes, vp]
    L.tq_dequantize.argtypes = [vp, Planes, i64, vp, i32, vp]
    L.tq_decode_workspace_bytes.argtypes = [vp, vp, i32, i32, i32, i32, ctypes.POINTER(sz)]
    L.tq_decode_attention.argtypes = [vp, vp, vp, i32, Planes, Planes, vp, i32, i32, i32, i32,
                                      ctypes.c_float, vp, vp, vp, sz, vp]
    L.tq_decode_attention_noalloc.argtypes = [vp, vp, vp, i32, Planes, Planes, vp, i32, i32, i32, i32,
                                              ctypes.c_float, vp, vp, vp]
    L.tq_decode_append_attention.argtypes = [vp, vp, vp, i32, vp, vp, i32, Planes, Planes, vp, i32, i32, i32, i32,
                                             ctypes.c_float, vp, vp, sz, vp]
    L.tq_select_outlier_channels.argtypes = [vp, i32, i64, i64, i32, i32, vp, vp, vp]
    L.tq_mixed_quantize.argtypes = [vp, vp, vp, vp, i32, i64, i64, Planes, Planes, vp, sz, vp]
    L.tq_mixed_quantize_kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, i64, Planes, Planes,
                                       Planes, Planes, vp, sz, vp]
    L.tq_mixed_quantize_scratch_bytes.argtypes = []
    L.tq_mixed_dequantize.argtypes = [vp, vp, vp, Planes, Planes, i64, vp, i32, vp]
    L.tq_mixed_decode_workspace_bytes.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, ctypes.POINTER(sz)]
    L.tq_mixed_decode_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, Planes, Planes, Planes, Planes, vp,
                                            i32, i32, i32, i32, ctypes.c_float, vp, vp, vp, sz, vp]
    L.tq_device_status.argtypes = [vp, ctypes.POINTER(i32), i32]
    L.tq_check_wait_timeout.argtypes = [vp, i32, u64, vp]
    L.tq_last_error.restype = ctypes.c_char_p
    for name in EXPORTED:
        if name != "tq_last_error":
            getattr(L, name).restype = i32
    L.tq_mixed_quantize_scratch_bytes.restype = sz
    _lib = L
    return L


def check(rc: int) -> None:
    if rc != TQ_OK:
        raise TQError(rc, lib().tq_last_error().decode(errors="replace"))
