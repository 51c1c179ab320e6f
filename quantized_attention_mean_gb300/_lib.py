"""ctypes declarations for libsageattn.so (the C ABI in include/sageattn.h).

Loading fails loudly when the library is missing: there is no fallback implementation.
"""

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsageattn.so")

c_int, c_float, c_size_t, c_int64, c_void_p = (ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                                                ctypes.c_int64, ctypes.c_void_p)


class SageTensor(ctypes.Structure):
    _fields_ = [("data", c_void_p), ("stride", c_int64 * 3)]


class SagePacked(ctypes.Structure):
    _fields_ = [("data", c_void_p), ("stride_token", c_int64), ("stride_head", c_int64)]


# name -> (restype, argtypes), mirroring include/sageattn.h
_T = ctypes.POINTER(SageTensor)
_P = ctypes.POINTER(SagePacked)
SIGNATURES = {
    "sage_attn_workspace_size": (c_size_t, [c_int] * 7),
    "sage_attn": (c_int, [_T, _T, _T, _T, c_void_p] + [c_int] * 9 + [c_float] + [c_int] * 5
                  + [c_void_p, c_size_t, c_void_p]),
    "sage_attn_qk_int8_pv_fp16": (c_int, [_T, _T, _T, _T, c_void_p] + [c_int] * 9 + [c_float]
                                  + [c_int] * 5 + [c_void_p, c_size_t, c_void_p]),
    "sage_attn_fp4": (c_int, [_T, _T, _T, _T, c_void_p] + [c_int] * 9 + [c_float]
                      + [c_int] * 5 + [c_void_p, c_size_t, c_void_p]),
    "sage_attn_no_alloc": (c_int, [_T, _T, _T, _T, c_void_p] + [c_int] * 9 + [c_float] + [c_int] * 5
                           + [c_void_p]),
    "sage_attn_varlen_workspace_size": (c_size_t, [c_int] * 7),
    "sage_attn_varlen": (c_int, [_P, _P, _P, _P, c_void_p, c_void_p, c_void_p] + [c_int] * 10
                         + [c_float] + [c_int] * 5 + [c_void_p, c_size_t, c_void_p]),
    "sage_attn_varlen_qk_int8_pv_fp16": (c_int, [_P, _P, _P, _P, c_void_p, c_void_p, c_void_p]
                                         + [c_int] * 10 + [c_float] + [c_int] * 5
                                         + [c_void_p, c_size_t, c_void_p]),
    "sage_status_string": (ctypes.c_char_p, [c_int]),
    "sage_last_cuda_error": (ctypes.c_char_p, []),
    "sage_read_device_status": (c_int, [c_void_p, c_void_p]),
    "sage_device_supported": (c_int, []),
    "sage_debug_export_quant": (c_int, [c_void_p] + [c_int] * 7 + [c_void_p] * 8 + [c_void_p]),
    "sage_attn_debug_scores": (c_int, [_T, _T, _T, _T, c_void_p] + [c_int] * 9 + [c_float]
                               + [c_int] * 5 + [c_void_p, c_size_t, c_void_p, c_void_p]),
    "sage_debug_e4m3": (c_int, [c_void_p, c_void_p, c_int64, c_void_p]),
    "sage_debug_e2m1": (c_int, [c_void_p, c_void_p, c_int64, c_void_p]),
    "sage_debug_export_fp16": (c_int, [c_void_p] + [c_int] * 7 + [c_void_p] * 3 + [c_void_p]),
    "sage_profile_enable": (c_int, [c_int]),
    "sage_debug_stall_attention": (c_int, [c_int]),
    "sage_debug_select_path": (c_int, [c_int]),
    "sage_debug_trace_attention": (c_int, [c_void_p]),
    "sage_profile_read": (c_int, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(c_int)]),
    # outs (array of sage_tensor), lses (array of float*), n, out, lse_out, B, H, N, d, dtype,
    # layout, stream
    "sage_merge_partials": (c_int, [c_void_p, c_void_p, c_int, _T, c_void_p] + [c_int] * 6
                            + [c_void_p]),
}

_lib = None


def load():
    """Returns the loaded library with typed entry points (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m quantized_attention_mean_gb300.build` "
            "(or __graft_entry__.build()); there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
