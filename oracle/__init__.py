"""CPU oracle for SageAttention-style quantized attention (test infrastructure).

This package is test infrastructure. Only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it. The product path (the CUDA library and its Python binding) never imports,
links or calls anything here, and nothing here imports the product package.
"""

from .sage_oracle import (  # noqa: F401
    E4M3_MAX,
    INT8_MAX,
    KV_TILE,
    QK_BLOCK,
    attention_emulated,
    attention_exact,
    bf16_round,
    e4m3_decode,
    e4m3_encode,
    key_mean_fp64,
    quantize_head,
    quantize_int8_blocks,
    quantize_v_channels,
    smooth_k_lse_term,
)
