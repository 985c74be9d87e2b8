"""Whole-tensor drivers of the oracle (test infrastructure only).

They loop the per-(batch, head) oracle functions over ``[B, S, H, D]`` ("NHD")
or ``[B, H, S, D]`` ("HND") float32 arrays holding bf16 values, and lay the
results out the way the library's quantize call writes them:

* Q and K codes: int8 ``[B, H, S_pad, D]``; rows ``S..S_pad-1`` are 0.
* Q and K scales: float32 ``[B, H, S_pad / 32]``; blocks past ``ceil(S/32)`` are 0.
* V codes, transposed: uint8 ``[B, H, D, S_pad]``; columns ``S..S_pad-1`` are 0.
* V scales and key means: float32 ``[B, H, D]``.

``S_pad`` rounds S up to a multiple of 128 (one key tile).
"""

from __future__ import annotations

import numpy as np

from .sage_oracle import (
    KV_TILE,
    QK_BLOCK,
    attention_emulated,
    attention_exact,
    e4m3_decode,
    quantize_head,
    smooth_k_lse_term,
)


def padded_len(s_len: int) -> int:
    return -(-s_len // KV_TILE) * KV_TILE


def head_view(x, layout: str, b: int, h: int) -> np.ndarray:
    """The [S, D] slice of one (batch, head)."""
    if layout == "NHD":
        return x[b, :, h, :]
    if layout == "HND":
        return x[b, h, :, :]
    raise ValueError(layout)


def dims(x, layout: str):
    if layout == "NHD":
        b, s, h, d = x.shape
    elif layout == "HND":
        b, h, s, d = x.shape
    else:
        raise ValueError(layout)
    return b, s, h, d


def quantize_tensors(q, k, v, layout: str = "NHD", smooth_k: bool = True, heads=None):
    """Oracle prologue over every (batch, head), in the library's output layouts.

    ``heads`` optionally restricts the work to a list of (b, h) pairs; the
    other entries are left as zeros.
    """
    bsz, s_len, n_h, d = dims(q, layout)
    s_pad = padded_len(s_len)
    n_blk = s_pad // QK_BLOCK
    out = dict(
        q_codes=np.zeros((bsz, n_h, s_pad, d), np.int8),
        k_codes=np.zeros((bsz, n_h, s_pad, d), np.int8),
        vt_codes=np.zeros((bsz, n_h, d, s_pad), np.uint8),
        q_scale=np.zeros((bsz, n_h, n_blk), np.float32),
        k_scale=np.zeros((bsz, n_h, n_blk), np.float32),
        v_scale=np.zeros((bsz, n_h, d), np.float32),
        k_mean=np.zeros((bsz, n_h, d), np.float32),
    )
    todo = [(b, h) for b in range(bsz) for h in range(n_h)] if heads is None else heads
    for b, h in todo:
        r = quantize_head(head_view(q, layout, b, h), head_view(k, layout, b, h),
                          head_view(v, layout, b, h), smooth_k)
        nb = r["q_scale"].shape[0]
        out["q_codes"][b, h, :s_len] = r["q_codes"]
        out["k_codes"][b, h, :s_len] = r["k_codes"]
        out["vt_codes"][b, h, :, :s_len] = r["v_codes"].T
        out["q_scale"][b, h, :nb] = r["q_scale"]
        out["k_scale"][b, h, :nb] = r["k_scale"]
        out["v_scale"][b, h] = r["v_scale"]
        out["k_mean"][b, h] = r["k_mean"]
    return out


def attention_from_codes(qz, s_len: int, sm_scale: float, b: int, h: int, rows=None,
                         return_fp32: bool = False, causal: bool = False, return_lse: bool = False,
                         q=None, layout: str = "NHD"):
    """Emulated attention of one (batch, head) from a quantized bundle
    laid out as :func:`quantize_tensors` returns it. With ``return_lse`` the
    pair (output, lse); when the bf16 query tensor ``q`` is given, the lse
    includes the smooth_k term from the bundle's key mean (the log-sum-exp of
    the original keys), otherwise it is that of the mean-reduced keys."""
    vt = qz["vt_codes"][b, h, :, :s_len]
    v_vals = e4m3_decode(vt.T)
    term = None
    if return_lse and q is not None:
        term = smooth_k_lse_term(head_view(q, layout, b, h), qz["k_mean"][b, h], sm_scale, rows=rows)
    return attention_emulated(qz["q_codes"][b, h, :s_len], qz["k_codes"][b, h, :s_len], v_vals,
                              qz["q_scale"][b, h], qz["k_scale"][b, h], qz["v_scale"][b, h],
                              sm_scale, rows=rows, return_fp32=return_fp32, causal=causal,
                              return_lse=return_lse, lse_term=term)


def exact_head(q, k, v, layout: str, sm_scale: float, b: int, h: int, rows=None, causal: bool = False,
               return_lse: bool = False):
    return attention_exact(head_view(q, layout, b, h), head_view(k, layout, b, h),
                           head_view(v, layout, b, h), sm_scale, rows=rows, causal=causal,
                           return_lse=return_lse)
