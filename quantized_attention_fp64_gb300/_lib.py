"""ctypes binding of libsage.so: loads the library and declares every entry
point of include/sage.h with its C signature. Argument marshalling only."""

from __future__ import annotations

import ctypes
import os
import re

from ._build import LIB_PATH, ROOT

c_i64 = ctypes.c_int64
c_int = ctypes.c_int
c_vp = ctypes.c_void_p
c_size_p = ctypes.POINTER(ctypes.c_size_t)
I64x4 = c_i64 * 4


class Bf16Tensor(ctypes.Structure):
    """sage_bf16_tensor"""
    _fields_ = [("ptr_dev", c_vp), ("stride_b", c_i64), ("stride_s", c_i64), ("stride_h", c_i64)]


class Quantized(ctypes.Structure):
    """sage_quantized"""
    _fields_ = [("q_codes_dev", c_vp), ("k_codes_dev", c_vp), ("vt_codes_dev", c_vp), ("q_scale_dev", c_vp),
                ("k_scale_dev", c_vp), ("v_scale_dev", c_vp), ("k_mean_dev", c_vp), ("q16_dev", c_vp),
                ("k16_dev", c_vp)]


class SageattnArgs(ctypes.Structure):
    """sage_sageattn_args"""
    _fields_ = [("q_dev", c_vp), ("k_dev", c_vp), ("v_dev", c_vp), ("q_shape", I64x4), ("k_shape", I64x4),
                ("v_shape", I64x4), ("q_strides", I64x4), ("k_strides", I64x4), ("v_strides", I64x4),
                ("out_strides", I64x4), ("q_dtype", ctypes.c_int32), ("k_dtype", ctypes.c_int32),
                ("v_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32), ("is_causal", ctypes.c_int32),
                ("smooth_k", ctypes.c_int32), ("sm_scale", ctypes.c_float), ("tensor_layout", ctypes.c_char * 4),
                ("out_dev", c_vp), ("lse_dev", c_vp), ("workspace_dev", c_vp), ("workspace_bytes", ctypes.c_size_t),
                ("cuda_stream", c_vp)]


_SIGNATURES = {
    "sage_bundle_size": (c_int, [c_i64, c_i64, c_i64, c_i64, c_size_p, c_vp, ctypes.POINTER(Quantized)]),
    "sage_quantize_scratch_size": (c_int, [c_i64, c_i64, c_i64, c_i64, c_size_p]),
    "sage_workspace_size": (c_int, [c_i64, c_i64, c_i64, c_i64, c_size_p]),
    "sage_quantize": (c_int, [ctypes.POINTER(Bf16Tensor)] * 3 + [c_i64, c_i64, c_i64, c_i64, c_int,
                                                                ctypes.POINTER(Quantized), c_vp, ctypes.c_size_t,
                                                                c_vp]),
    "sage_quantize_noalloc": (c_int, [ctypes.POINTER(Bf16Tensor)] * 3 + [c_i64, c_i64, c_i64, c_i64, c_int,
                                                                        ctypes.POINTER(Quantized), c_vp]),
    "sage_attention": (c_int, [ctypes.POINTER(Quantized), c_i64, c_i64, c_i64, c_i64, ctypes.c_float, c_vp,
                               c_i64, c_i64, c_i64, c_vp]),
    "sage_attention_ex": (c_int, [ctypes.POINTER(Quantized), c_i64, c_i64, c_i64, c_i64, ctypes.c_float, c_int,
                                  c_vp, c_i64, c_i64, c_i64, c_vp, c_vp]),
    "sage_attention_simt": (c_int, [ctypes.POINTER(Quantized), c_i64, c_i64, c_i64, c_i64, ctypes.c_float, c_int,
                                    c_vp, c_i64, c_i64, c_i64, c_vp, c_vp]),
    "sage_lse_smooth_k_term": (c_int, [ctypes.POINTER(Bf16Tensor), c_vp, c_i64, c_i64, c_i64, c_i64, ctypes.c_float,
                                       c_vp, c_vp]),
    "sage_sageattn": (c_int, [c_vp, c_vp, c_vp, I64x4, I64x4, I64x4, I64x4, I64x4, I64x4, c_int, c_int, c_int,
                              ctypes.c_char_p, c_int, ctypes.c_float, c_int, c_int, c_vp, I64x4, c_int, c_vp,
                              ctypes.c_size_t, c_vp]),
    "sage_sageattn_ex": (c_int, [c_vp, c_vp, c_vp, I64x4, I64x4, I64x4, I64x4, I64x4, I64x4, c_int, c_int, c_int,
                                 ctypes.c_char_p, c_int, ctypes.c_float, c_int, c_vp, I64x4, c_int, c_vp, c_vp,
                                 ctypes.c_size_t, c_vp]),
    "sage_sageattn_args_call": (c_int, [ctypes.POINTER(SageattnArgs)]),
    "sage_host_workspace_size": (c_int, [c_i64, c_i64, c_i64, c_i64, c_int, c_size_p]),
    "sage_sageattn_host": (c_int, [c_vp, c_vp, c_vp, I64x4, c_int, ctypes.c_char_p, c_int, ctypes.c_float, c_int, c_vp,
                                   c_int, c_vp, ctypes.c_size_t, c_vp]),
    "sage_device_error": (c_int, [c_vp, ctypes.POINTER(c_int)]),
    "sage_selftest_wait_timeout": (c_int, [c_vp]),
    "sage_strerror": (ctypes.c_char_p, [c_int]),
}

_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/sage.h declares."""
    with open(os.path.join(ROOT, "include", "sage.h")) as f:
        text = f.read()
    return re.findall(r"SAGE_API\s+(?:const\s+)?\w+\s*\*?\s*(sage_\w+)\s*\(", text)


def ensure_built() -> str:
    from ._build import build

    return build()


def load():
    """Load libsage.so (it must have been built) and declare its signatures."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with quantized_attention_fp64_gb300._build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
