"""Pins for the oracle at head dimension 64 (the second workload of the pages:
"Hand-written prologue ... (v0.4.0)", section "Worth knowing", and the
kernels-community issue's note that head_dim 64 is not covered yet).

The oracle's functions take the head dimension from their inputs; these pins
check that nothing in them assumes 128: brute force of the INT8 blocks (32
tokens x 64 channels) with exact rationals, the fp64 key mean against
math.fsum, exact attention against Python loops, and the emulation against
exact attention without quantization and at the accuracy the method reaches.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import (attention_emulated, attention_exact, e4m3_decode, key_mean_fp64, quantize_head,
                    quantize_int8_blocks, quantize_v_channels)

D = 64
SM64 = np.float32(1.0 / math.sqrt(64.0))


def _round_bf16(x):
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(np.float32)


def _bf16(rng, shape, scale=1.0):
    return _round_bf16(rng.standard_normal(shape) * scale)


def test_int8_blocks_bruteforce_d64():
    rng = np.random.default_rng(64)
    x = _bf16(rng, (70, D), 2.0)
    codes, scales = quantize_int8_blocks(x)
    assert codes.shape == (70, D) and scales.shape == (3,)
    for t in range(3):
        blk = x[32 * t:32 * (t + 1)]
        a = np.float32(np.abs(blk).max())
        assert scales[t] == np.float32(a / np.float32(127))
        s = Fraction(float(scales[t]))
        for r in range(blk.shape[0]):
            for c in range(D):
                q = float(np.float32(blk[r, c] / scales[t]))   # fl32(x / s)
                assert codes[32 * t + r, c] == round(q)        # round half even (Python round)
                # within half a step, up to the rounding of the quotient x / s
                # (fl32(x / s) is within half an ulp of 127.5 or less: 2^-18)
                assert abs(Fraction(float(blk[r, c])) - codes[32 * t + r, c] * s) <= s * (Fraction(1, 2) + Fraction(1, 2 ** 17))


def test_key_mean_d64_matches_fsum():
    rng = np.random.default_rng(65)
    k = _bf16(rng, (1000, D), 3.0)
    mean = key_mean_fp64(k)
    ref = np.array([math.fsum(float(v) for v in k[:, c]) / 1000 for c in range(D)])
    assert np.array_equal(mean, ref.astype(np.float32))


def test_v_channels_d64():
    rng = np.random.default_rng(66)
    v = _bf16(rng, (300, D))
    codes, scales = quantize_v_channels(v)
    assert codes.shape == (300, D) and scales.shape == (D,)
    dec = e4m3_decode(codes).astype(np.float64) * scales[None, :]
    assert np.all(np.abs(dec - v) <= np.abs(v) * 2.0 ** -4 + scales[None, :] * 2.0 ** -10)
    # every channel's largest magnitude maps to +-448
    assert np.all(np.abs(e4m3_decode(codes)).max(axis=0) == 448.0)


@pytest.mark.parametrize("causal", [False, True])
def test_exact_d64_bruteforce(causal):
    rng = np.random.default_rng(67)
    s_len = 6
    q, k, v = (_bf16(rng, (s_len, D)) for _ in range(3))
    out, lse = attention_exact(q, k, v, SM64, causal=causal, return_lse=True)
    for i in range(s_len):
        keys = range(i + 1) if causal else range(s_len)
        logits = [float(SM64) * math.fsum(float(q[i, c]) * float(k[j, c]) for c in range(D)) for j in keys]
        mx = max(logits)
        w = [math.exp(t - mx) for t in logits]
        z = math.fsum(w)
        assert abs(lse[i] - (mx + math.log(z))) <= 1e-12 * max(1.0, abs(mx))
        for c in range(D):
            ref = math.fsum(wj * float(v[j, c]) for wj, j in zip(w, keys)) / z
            assert abs(out[i, c] - ref) <= 1e-12


@pytest.mark.parametrize("s_len", [1, 129, 300])
def test_emulation_d64_reduces_to_exact_without_quantization(s_len):
    rng = np.random.default_rng(s_len + 68)
    q, k, v = (_bf16(rng, (s_len, D), 1.5) for _ in range(3))
    nb = -(-s_len // 32)
    ones = np.ones(nb, np.float32)
    got = attention_emulated(q, k, v, ones, ones, np.ones(D, np.float32), SM64, quantize_p=False,
                             return_fp32=True)
    ref = attention_exact(q, k, v, SM64)
    assert np.abs(got - ref).max() <= 2e-5 * np.abs(ref).max()


@pytest.mark.parametrize("smooth", [False, True])
def test_emulation_d64_accuracy(smooth):
    rng = np.random.default_rng(69 + smooth)
    s_len = 1000
    q, v = _bf16(rng, (s_len, D)), _bf16(rng, (s_len, D))
    k = _round_bf16(rng.standard_normal((s_len, D)) + rng.standard_normal(D)[None, :] * 2.0)
    r = quantize_head(q, k, v, smooth_k=smooth)
    assert r["q_codes"].shape == (s_len, D) and r["k_mean"].shape == (D,)
    emu = attention_emulated(r["q_codes"], r["k_codes"], e4m3_decode(r["v_codes"]), r["q_scale"], r["k_scale"],
                             r["v_scale"], SM64)
    ref = attention_exact(q, k, v, SM64)
    a, b = emu.astype(np.float64).ravel(), ref.ravel()
    assert a @ b / (np.linalg.norm(a) * np.linalg.norm(b)) >= 0.999
