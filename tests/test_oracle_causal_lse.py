"""Pins for the oracle's causal mask and log-sum-exp (the `is_causal` and
`return_lse` flags of the sageattn entry).

References: pure-Python brute force (math.exp / math.fsum) on tiny inputs;
closed forms (the first row sees one key, a zero query averages the visible
values, the last causal row is the unmasked row); the exact identity that a
per-channel key shift moves every logit of a row by sm_scale * q . shift;
reduction of the emulation to exact attention when every quantization is the
identity; and the equivalence of skipping fully masked key tiles, which the
kernel relies on.
"""

import math

import numpy as np
import pytest

from oracle import attention_emulated, attention_exact, e4m3_decode, quantize_head, smooth_k_lse_term

SM = np.float32(1.0 / math.sqrt(128.0))


def _round_bf16(x):
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(np.float32)


def _bf16(rng, shape, scale=1.0):
    return _round_bf16(rng.standard_normal(shape) * scale)


@pytest.mark.parametrize("s_len,d,causal", [(1, 4, True), (3, 4, True), (9, 5, True), (7, 3, False)])
def test_exact_causal_lse_bruteforce(s_len, d, causal):
    rng = np.random.default_rng(s_len * 7 + d)
    q, k, v = (_bf16(rng, (s_len, d)) for _ in range(3))
    sm = float(np.float32(0.41))
    out, lse = attention_exact(q, k, v, sm, causal=causal, return_lse=True)
    for i in range(s_len):
        keys = range(i + 1) if causal else range(s_len)
        logits = [sm * math.fsum(float(q[i, c]) * float(k[j, c]) for c in range(d)) for j in keys]
        mx = max(logits)
        w = [math.exp(t - mx) for t in logits]
        z = math.fsum(w)
        assert abs(lse[i] - (mx + math.log(z))) <= 1e-12 * max(1.0, abs(mx))
        for c in range(d):
            ref = math.fsum(wj * float(v[j, c]) for wj, j in zip(w, keys)) / z
            assert abs(out[i, c] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_exact_causal_closed_forms():
    rng = np.random.default_rng(21)
    s_len = 300
    q, k, v = (_bf16(rng, (s_len, 128)) for _ in range(3))
    out, lse = attention_exact(q, k, v, SM, causal=True, return_lse=True)
    # the first row sees only key 0
    assert np.abs(out[0] - v[0]).max() <= 1e-15
    assert abs(lse[0] - float(SM) * float(q[0].astype(np.float64) @ k[0].astype(np.float64))) <= 1e-12
    # the last row sees every key: it is the unmasked row
    full, full_lse = attention_exact(q, k, v, SM, rows=[s_len - 1], return_lse=True)
    assert np.abs(out[-1] - full[0]).max() <= 1e-12 and abs(lse[-1] - full_lse[0]) <= 1e-12
    # a zero query weighs the visible keys equally: the running mean of V, lse = ln(i + 1)
    zq = np.zeros_like(q)
    out0, lse0 = attention_exact(zq, k, v, SM, causal=True, return_lse=True)
    mean = np.cumsum(v.astype(np.float64), axis=0) / np.arange(1, s_len + 1)[:, None]
    assert np.abs(out0 - mean).max() <= 1e-12
    assert np.abs(lse0 - np.log(np.arange(1, s_len + 1))).max() <= 1e-12


def test_exact_lse_key_shift_identity():
    # Shifting every key by the same per-channel vector mu leaves the output
    # unchanged and moves row i's log-sum-exp by exactly sm_scale * q_i . mu;
    # this is the term the quantized path adds back when smooth_k is on.
    rng = np.random.default_rng(22)
    q, v = _bf16(rng, (200, 128)), _bf16(rng, (200, 128))
    k = (np.round(rng.standard_normal((200, 128)) * 64.0) / 64.0).astype(np.float32)
    # keys on a 1/64 grid, shifts on a 1/8 grid: every shifted key is exact in fp32
    mu = np.round(rng.standard_normal(128) * 24.0) / 8.0
    shifted = k.astype(np.float64) + mu
    assert np.array_equal(shifted.astype(np.float32).astype(np.float64), shifted)
    for causal in (False, True):
        o1, l1 = attention_exact(q, k, v, SM, causal=causal, return_lse=True)
        o2, l2 = attention_exact(q, shifted.astype(np.float32), v, SM, causal=causal, return_lse=True)
        shift = float(SM) * (q.astype(np.float64) @ mu)
        assert np.abs(o1 - o2).max() <= 1e-10
        assert np.abs((l2 - l1) - shift).max() <= 1e-9 * max(1.0, np.abs(shift).max())


@pytest.mark.parametrize("s_len", [1, 100, 129, 300])
def test_emulation_causal_reduces_to_exact_without_quantization(s_len):
    rng = np.random.default_rng(s_len + 40)
    q, k, v = (_bf16(rng, (s_len, 128), 1.5) for _ in range(3))
    nb = -(-s_len // 32)
    ones = np.ones(nb, np.float32)
    got, lse = attention_emulated(q, k, v, ones, ones, np.ones(128, np.float32), SM, quantize_p=False,
                                  return_fp32=True, causal=True, return_lse=True)
    ref, ref_lse = attention_exact(q, k, v, SM, causal=True, return_lse=True)
    assert np.abs(got - ref).max() <= 2e-5 * np.abs(ref).max()
    # lse = m + ln(l) with l summing p = exp(logit - m) over the visible keys
    assert np.abs(lse - ref_lse).max() <= 1e-5 * max(1.0, np.abs(ref_lse).max())


def test_emulation_causal_skipping_masked_tiles_is_exact():
    # A kernel skips the key tiles a row cannot see. Row i's result from only
    # the keys up to the end of its own tile must equal, bit for bit, its
    # result over every key with the mask applied (a fully masked tile has
    # alpha = 1 and p = 0).
    rng = np.random.default_rng(23)
    s_len = 517
    q, k, v = (_bf16(rng, (s_len, 128)) for _ in range(3))
    r = quantize_head(q, k, v, smooth_k=True)
    vv = e4m3_decode(r["v_codes"])
    full, full_lse = attention_emulated(r["q_codes"], r["k_codes"], vv, r["q_scale"], r["k_scale"], r["v_scale"],
                                        SM, causal=True, return_lse=True)
    for i in (0, 5, 127, 128, 300, 516):
        end = min(s_len, (i // 128 + 1) * 128)
        part, part_lse = attention_emulated(r["q_codes"], r["k_codes"][:end], vv[:end], r["q_scale"], r["k_scale"],
                                            r["v_scale"], SM, rows=[i], causal=True, return_lse=True)
        assert np.array_equal(part[0], full[i]) and part_lse[0] == full_lse[i]


@pytest.mark.parametrize("causal", [False, True])
def test_emulated_lse_needs_and_gets_the_smooth_k_term(causal):
    # Keys with large channel offsets, smooth_k on: the emulated log-sum-exp
    # tracks the exact one only with the key-mean term added back, and with
    # the term taken from the bf16 query it is more accurate than without
    # smoothing (whose error is that of the quantized logits).
    rng = np.random.default_rng(24 + causal)
    s_len = 700
    q, v = _bf16(rng, (s_len, 128)), _bf16(rng, (s_len, 128))
    k = _round_bf16(rng.standard_normal((s_len, 128)) + rng.standard_normal(128)[None, :] * 3.0)
    r = quantize_head(q, k, v, smooth_k=True)
    args = (r["q_codes"], r["k_codes"], e4m3_decode(r["v_codes"]), r["q_scale"], r["k_scale"], r["v_scale"], SM)
    term = smooth_k_lse_term(q, r["k_mean"], SM)
    _, lse = attention_emulated(*args, causal=causal, return_lse=True, lse_term=term)
    _, lse_no_term = attention_emulated(*args, causal=causal, return_lse=True)
    _, ref = attention_exact(q, k, v, SM, causal=causal, return_lse=True)
    r0 = quantize_head(q, k, v, smooth_k=False)
    _, lse0 = attention_emulated(r0["q_codes"], r0["k_codes"], e4m3_decode(r0["v_codes"]), r0["q_scale"],
                                 r0["k_scale"], r0["v_scale"], SM, causal=causal, return_lse=True)
    err, err_off = np.abs(lse - ref), np.abs(lse0 - ref)
    assert np.abs(lse_no_term - ref).max() >= 0.5
    assert err.max() <= 0.05 and err.mean() <= 0.5 * err_off.mean()
    # the term itself: sm_scale * q . mean, against a plain Python sum
    for i in (0, 350, 699):
        ref_t = float(SM) * math.fsum(float(q[i, c]) * float(r["k_mean"][c]) for c in range(128))
        assert abs(term[i] - ref_t) <= 1e-12 * max(1.0, abs(ref_t))
