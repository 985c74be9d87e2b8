"""Plain CPU oracle for SageAttention-style quantized attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. It shares no code, header, table or constant with the CUDA library, and
it imports nothing from the product package.

What it computes, and where each step comes from
------------------------------------------------
Sources (web pages; cited by title and section):

* [IX] "aiter-sage-attention: SageAttention for AMD RDNA4 (gfx1201) #1222"
  (huggingface/kernels-community issue), section "The kernel": QK^T is
  computed in INT8 and PV in FP8, both with FP32 accumulation; Q and K are
  quantized per 32-row block and V per channel. Section "What I have so far":
  the ``sageattn(q, k, v, tensor_layout, is_causal, sm_scale, return_lse)``
  entry, its rejections, and the cosine of 0.9992 against SDPA.
* [RN] "Hand-written prologue: faster short calls, no compiler, RX 9060 XT
  opt-in (v0.4.0)" (SageAttention-RDNA4 release notes), section "What
  changed": with smooth_k on, the key mean is summed in fp64; the prologue
  uses 64-bit offsets so there is no sequence-length ceiling.
* [CA] "gfx1201 (RDNA4) SageAttention attention backend: aiter package or Hub
  kernel?", section "原因分析" (cause analysis): inputs are BF16
  ``[B, S, H, 128]``, Q/K/V of one shape, no mask, not causal.

Where the pages leave a step open, this module takes one reading, stated at
the function that uses it (the full list is kept with the design notes):
round-half-even INT8 codes in +-127; scale = amax/127 unscaled by sm_scale;
x/scale correctly rounded in fp32; the fp64 key sum in a fixed order (each
32-token chunk left to right from +0.0, then a pairwise tree over chunks);
V scaled per channel over all tokens to the OCP e4m3fn maximum 448 with
round-half-even and saturation; online softmax over 128-key tiles in
ascending order, always rescaling with the exact running maximum; P quantized
as e4m3(448 * p) and the row sum taken from the unquantized fp32 p.

Parity pins that hold this module to something other than itself live in
``tests/test_oracle_*.py``.
"""

from __future__ import annotations

import math

import numpy as np

QK_BLOCK = 32      # tokens per Q/K scale block ([IX] "The kernel": per 32-row block)
INT8_MAX = 127     # symmetric int8 code range; -128 is never produced (reading)
E4M3_MAX = 448.0   # largest finite value of OCP FP8 E4M3 ("e4m3fn")
KV_TILE = 128      # keys per online-softmax step (reading)
P_SCALE = 448.0    # p in [0, 1] is stored as e4m3(448 * p) (reading)

_F32 = np.float32
_F64 = np.float64


# ----------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    """Round float32 values to the nearest bfloat16, ties to even.

    bfloat16 keeps the top 16 bits of a float32. Rounding to nearest even adds
    0x7FFF plus the lowest kept bit to the 32-bit pattern and truncates. NaN
    stays NaN. Returns float32 values that are exactly representable in bf16.
    """
    x = np.ascontiguousarray(x, dtype=_F32)
    u = x.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)) << np.uint64(16)
    out = r.astype(np.uint32).view(_F32).copy()
    out[np.isnan(x)] = np.nan
    return out


def _e4m3_value_table() -> np.ndarray:
    """Value of each of the 256 OCP E4M3 ("e4m3fn") codes, from the format.

    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits. Exponent field 0
    holds the subnormals m * 2^-9. The pattern S.1111.111 is NaN; there are no
    infinities, so the largest finite magnitude is 1.75 * 2^8 = 448.
    """
    vals = np.empty(256, dtype=_F64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = math.nan
        elif e == 0:
            vals[code] = sign * m * 2.0 ** -9
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3_VALUES = _e4m3_value_table()


def e4m3_decode(codes) -> np.ndarray:
    """Values (float32, exact) of e4m3fn codes (uint8)."""
    return _E4M3_VALUES[np.asarray(codes, dtype=np.uint8)].astype(_F32)


def e4m3_encode(x) -> np.ndarray:
    """Encode float32 values as e4m3fn codes, round half to even, saturating.

    Reading: the rounding is round-to-nearest-even and values beyond the
    largest finite magnitude 448 saturate to +-448 (no format has infinities;
    "satfinite"). The sign of zero is kept. NaN maps to the NaN code.

    Method: in float64 (exact for every step below), find the binade exponent
    e = floor(log2 |x|), clamped to [-6, 8] (below -6 every value shares the
    subnormal spacing 2^-9), round |x| to a multiple of the spacing 2^(e-3)
    with ties to even, clamp to 448, then write the code fields.
    """
    x = np.asarray(x, dtype=_F32)
    a = np.abs(x.astype(_F64))
    neg = np.signbit(x)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, a)
    with np.errstate(over="ignore", invalid="ignore"):
        _, k = np.frexp(a)                     # a = f * 2^k with f in [0.5, 1)
        e = np.clip(k - 1, -6, 8)
        spacing = np.ldexp(1.0, e - 3)
        r = np.rint(a / spacing) * spacing     # exact quotient, ties to even
        r = np.where(np.isinf(a), E4M3_MAX, r)
        r = np.minimum(r, E4M3_MAX)
    sub = r < 2.0 ** -6
    code_sub = np.rint(r / 2.0 ** -9)
    _, k2 = np.frexp(np.where(sub, 1.0, r))
    big_e = k2 - 1
    mant = np.where(sub, 0.0, r / np.ldexp(1.0, big_e) * 8.0 - 8.0)
    code_norm = (big_e + 7) * 8 + mant
    code = np.where(sub, code_sub, code_norm).astype(np.int64)
    code = np.where(nan, 0x7F, code)
    code = code | (neg.astype(np.int64) << 7)
    return code.astype(np.uint8)


# ----------------------------------------------------------------------------
# Prologue: key mean, INT8 Q/K blocks, FP8 V channels
# ----------------------------------------------------------------------------

def key_mean_fp64(k32) -> np.ndarray:
    """Per-channel mean of the keys of one (batch, head), summed in fp64.

    [RN] "What changed": with smooth_k on, the key mean is summed in fp64.
    Reading of the order (the page gives none): the tokens are cut into
    chunks of 32; each chunk is summed left to right in fp64 starting from
    +0.0; the chunk sums are combined by a pairwise tree (pad the list to a
    power of two with +0.0, then repeatedly add neighbours 2i and 2i+1). The
    total T is divided by S in fp64 and rounded once to fp32.

    k32: float32 [S, D] (bf16 values). Returns float32 [D].
    """
    k32 = np.asarray(k32, dtype=_F32)
    s_len, d = k32.shape
    n_chunks = -(-s_len // QK_BLOCK)
    partial = np.zeros((n_chunks, d), dtype=_F64)
    for c in range(n_chunks):
        acc = np.zeros(d, dtype=_F64)
        for s in range(c * QK_BLOCK, min((c + 1) * QK_BLOCK, s_len)):
            acc = acc + k32[s].astype(_F64)
        partial[c] = acc
    width = 1
    while width < n_chunks:
        width *= 2
    level = np.zeros((width, d), dtype=_F64)
    level[:n_chunks] = partial
    while level.shape[0] > 1:
        level = level[0::2] + level[1::2]
    total = level[0]
    return (total / _F64(s_len)).astype(_F32)


def quantize_int8_blocks(x32):
    """Symmetric INT8 codes for one (batch, head), one scale per 32 tokens.

    [IX] "The kernel": Q and K are quantized per 32-row block. Readings: a
    block is 32 consecutive tokens with all channels (the last block may be
    short and uses only its valid rows); the scale is s = amax / 127 in fp32;
    a code is rint(x / s) with x / s correctly rounded in fp32 and ties to
    even, clamped to [-127, 127]; an all-zero block has s = 0 and codes 0.

    x32: float32 [S, D]. Returns (codes int8 [S, D], scales float32 [ceil(S/32)]).
    """
    x32 = np.asarray(x32, dtype=_F32)
    s_len, d = x32.shape
    n_blk = -(-s_len // QK_BLOCK)
    codes = np.zeros((s_len, d), dtype=np.int8)
    scales = np.zeros(n_blk, dtype=_F32)
    for t in range(n_blk):
        blk = x32[t * QK_BLOCK:min((t + 1) * QK_BLOCK, s_len)]
        amax = _F32(np.max(np.abs(blk)))
        if amax == 0:
            continue
        s = _F32(amax / _F32(INT8_MAX))
        q = (blk / s).astype(_F32)
        codes[t * QK_BLOCK:t * QK_BLOCK + blk.shape[0]] = np.clip(np.rint(q), -INT8_MAX, INT8_MAX).astype(np.int8)
        scales[t] = s
    return codes, scales


def quantize_v_channels(v32):
    """FP8 e4m3 codes for the values of one (batch, head), one scale per channel.

    [IX] "The kernel": V is quantized per channel. Readings: a channel's scale
    covers all S tokens, s_v = amax / 448 in fp32; a code is
    e4m3(v / s_v) with v / s_v correctly rounded in fp32; an all-zero channel
    has s_v = 0 and codes 0.

    v32: float32 [S, D]. Returns (codes uint8 [S, D] token-major, scales float32 [D]).
    """
    v32 = np.asarray(v32, dtype=_F32)
    amax = np.max(np.abs(v32), axis=0).astype(_F32)
    scales = (amax / _F32(E4M3_MAX)).astype(_F32)
    codes = np.zeros(v32.shape, dtype=np.uint8)
    live = scales > 0
    if np.any(live):
        q = (v32[:, live] / scales[live][None, :]).astype(_F32)
        codes[:, live] = e4m3_encode(q)
    return codes, scales


def quantize_head(q32, k32, v32, smooth_k: bool):
    """The whole prologue for one (batch, head).

    smooth_k ([RN] "What changed"): the per-channel key mean is subtracted
    from every key in fp32 (k' = fl(k - mean)) before INT8 quantization. It
    applies to K only (reading). With smooth_k off the mean is not computed
    and reported as 0.
    """
    k32 = np.asarray(k32, dtype=_F32)
    if smooth_k:
        mean = key_mean_fp64(k32)
        k_used = (k32 - mean[None, :]).astype(_F32)
    else:
        mean = np.zeros(k32.shape[1], dtype=_F32)
        k_used = k32
    q_codes, q_scale = quantize_int8_blocks(q32)
    k_codes, k_scale = quantize_int8_blocks(k_used)
    v_codes, v_scale = quantize_v_channels(v32)
    return dict(q_codes=q_codes, q_scale=q_scale, k_codes=k_codes, k_scale=k_scale,
                v_codes=v_codes, v_scale=v_scale, k_mean=mean)


# ----------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------

def _visible(rows, j0, j1, causal):
    """Key mask of one tile for the selected query rows: True where key j may
    be attended to. Without a mask every key is visible; with the causal mask
    query i sees keys j <= i (Q and K have the same length, so the mask is
    the lower triangle)."""
    if not causal:
        return None
    return np.arange(j0, j1)[None, :] <= np.asarray(rows)[:, None]


def attention_emulated(q_codes, k_codes, v_vals, q_scale, k_scale, v_scale, sm_scale,
                       rows=None, quantize_p: bool = True, return_fp32: bool = False,
                       causal: bool = False, return_lse: bool = False, lse_term=None):
    """Quantized flash attention for one (batch, head), emulated step by step.

    [IX] "The kernel": QK^T in INT8 with 32-bit integer accumulation, PV in
    FP8 with FP32 accumulation. Per query row and per tile of 128 keys, in
    ascending key order (reading):

    1. S_ij = sum_d qc_id * kc_jd, exact integers.
    2. logit_ij = fl32(S_ij) * c_ij, c_ij = (s_q[i/32] * s_k[j/32]) * sm_scale (fp32);
       keys the causal mask hides get -inf.
    3. m' = max(m, max_j logit_ij); alpha = exp(m - m'); p_ij = exp(logit_ij - m')
       (the differences in fp32, exp evaluated in fp64 and rounded to fp32).
    4. l = alpha * l + sum_j p_ij, from the unquantized p (tile sum in fp64,
       rounded to fp32).
    5. p~_ij = e4m3(448 * p_ij) (skipped when ``quantize_p`` is False).
    6. acc_d = alpha * acc_d + fl32(sum_j dec(p~_ij) * v_jd); the tile sum of
       products of two e4m3 values is exact in fp64.
    7. m = m'.

    Finally O_id = ((acc_d / l) * s_v[d]) / 448 in fp32, rounded to bf16.

    A tile the causal mask hides completely leaves m, l and acc unchanged
    (alpha = 1, p = 0), so skipping it, as a kernel does, gives the same
    result.

    Log-sum-exp (``return_lse``; the pages name the flag, not its meaning).
    Reading: the natural log of sum_j exp(sm_scale * q_i . k_j) over the keys
    row i sees, as fp32, which is what lets partial attention results over
    disjoint key sets be merged. From the emulation it is m + ln(l), the
    log-sum-exp of the logits of the codes. The K codes are of k - mean when
    smooth_k is on; a per-channel key shift changes every logit of row i by
    the same sm_scale * q_i . mean, so ``lse_term`` (see smooth_k_lse_term)
    is added to restore the log-sum-exp of the original keys:
    lse_i = m_i + ln(l_i) + lse_term_i, in fp64, rounded to fp32.

    q_codes, k_codes: [S, D] integer codes (or float values for the
    identity-quantization pin); v_vals: float32 [S, D] decoded V codes;
    q_scale, k_scale: float32 [ceil(S/32)]; v_scale: float32 [D].
    Returns bf16-rounded float32 [R, D] for the selected query rows, or the
    fp32 values before that rounding when ``return_fp32``; with
    ``return_lse`` a pair (output, lse float32 [R]).
    """
    k_codes = np.asarray(k_codes)
    s_len, d = k_codes.shape
    rows = np.arange(np.asarray(q_codes).shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    n_rows = rows.shape[0]
    qc = np.asarray(q_codes)[rows].astype(_F64)
    sq = np.asarray(q_scale, dtype=_F32)[rows // QK_BLOCK]
    sk = np.asarray(k_scale, dtype=_F32)
    sv = np.asarray(v_scale, dtype=_F32)
    v_vals = np.asarray(v_vals, dtype=_F32)
    scale = _F32(sm_scale)
    m = np.full(n_rows, -np.inf, dtype=_F32)
    l = np.zeros(n_rows, dtype=_F32)
    acc = np.zeros((n_rows, d), dtype=_F32)
    for j0 in range(0, s_len, KV_TILE):
        j1 = min(j0 + KV_TILE, s_len)
        s_ij = qc @ k_codes[j0:j1].astype(_F64).T
        c = ((sq[:, None] * sk[np.arange(j0, j1) // QK_BLOCK][None, :]).astype(_F32) * scale).astype(_F32)
        logit = (s_ij.astype(_F32) * c).astype(_F32)
        vis = _visible(rows, j0, j1, causal)
        if vis is not None:
            logit = np.where(vis, logit, _F32(-np.inf)).astype(_F32)
        m_new = np.maximum(m, logit.max(axis=1))
        with np.errstate(invalid="ignore"):
            alpha = np.exp((m - m_new).astype(_F64)).astype(_F32)
        alpha = np.where(m == m_new, _F32(1.0), alpha).astype(_F32)  # also for -inf - (-inf)
        p = np.exp((logit - m_new[:, None]).astype(_F32).astype(_F64)).astype(_F32)
        l = (alpha * l + p.astype(_F64).sum(axis=1).astype(_F32)).astype(_F32)
        p448 = (_F32(P_SCALE) * p).astype(_F32)
        p_used = e4m3_decode(e4m3_encode(p448)) if quantize_p else p448
        pv = (p_used.astype(_F64) @ v_vals[j0:j1].astype(_F64)).astype(_F32)
        acc = (alpha[:, None] * acc + pv).astype(_F32)
        m = m_new
    out = ((((acc / l[:, None]).astype(_F32)) * sv[None, :]).astype(_F32) / _F32(P_SCALE)).astype(_F32)
    out = out if return_fp32 else bf16_round(out)
    if not return_lse:
        return out
    term = np.zeros(n_rows, dtype=_F64) if lse_term is None else np.asarray(lse_term, dtype=_F64)
    lse = (m.astype(_F64) + np.log(l.astype(_F64)) + term).astype(_F32)
    return out, lse


def smooth_k_lse_term(q32, k_mean, sm_scale, rows=None) -> np.ndarray:
    """The log-sum-exp term of smooth_k: sm_scale * q_i . mean for each query
    row, with the bf16 query values (not their codes, which would add the Q
    quantization error) and the fp32 key mean, in fp64. Zero when the mean is
    zero (smooth_k off)."""
    q32 = np.asarray(q32, dtype=_F32)
    rows = np.arange(q32.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    return _F64(_F32(sm_scale)) * (q32[rows].astype(_F64) @ np.asarray(k_mean, dtype=_F32).astype(_F64))


def attention_exact(q32, k32, v32, sm_scale, rows=None, causal: bool = False, return_lse: bool = False):
    """Exact softmax attention in fp64 for one (batch, head), no quantization.

    O = softmax(sm_scale * Q K^T) V over all S keys ([CA] "原因分析": no mask,
    not causal), or with ``causal`` over the keys j <= i, with the logits,
    the two-pass softmax and the product with V all in fp64. Inputs are the
    bf16 values as float32 [S, D]. With ``return_lse`` also the natural-log
    log-sum-exp of each row's logits (fp64).
    """
    q32 = np.asarray(q32, dtype=_F32)
    rows = np.arange(q32.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    qf = q32[rows].astype(_F64)
    kf = np.asarray(k32, dtype=_F32).astype(_F64)
    vf = np.asarray(v32, dtype=_F32).astype(_F64)
    logits = (qf @ kf.T) * _F64(_F32(sm_scale))
    if causal:
        logits = np.where(np.arange(kf.shape[0])[None, :] <= rows[:, None], logits, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    z = p.sum(axis=1, keepdims=True)
    out = (p @ vf) / z
    if return_lse:
        return out, (m + np.log(z))[:, 0]
    return out
