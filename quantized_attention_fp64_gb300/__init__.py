"""GB300 (sm_103a) SageAttention-style quantized attention.

The computation lives in the CUDA library ``libsage.so`` (C ABI declared in
``include/sage.h``); this package loads it with ctypes and marshals torch
tensors into it. Build the library with ``quantized_attention_fp64_gb300._build.build()``.
"""

from .api import (  # noqa: F401
    QuantizedQKV,
    SageError,
    alloc_bundle,
    attention,
    attention_simt,
    device_error,
    host_workspace_size,
    lse_smooth_k_term,
    quantize,
    quantize_scratch_size,
    release_workspace_cache,
    sageattn,
    sageattn_ex,
    sageattn_host,
    workspace_size,
)
