"""Pins for the oracle's prologue: fp64 key mean, INT8 Q/K blocks, FP8 V channels.

The references here are exact rational arithmetic (``fractions``), math.fsum,
brute-force search over the e4m3 value set, hand-derived cases for the
summation-order reading, and invariants the method fixes.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import (E4M3_MAX, INT8_MAX, QK_BLOCK, e4m3_decode, key_mean_fp64, quantize_head,
                    quantize_int8_blocks, quantize_v_channels)
from oracle.tensors import quantize_tensors
from pin_util import e4m3_round_bruteforce, f32_round, round_half_even


def _bf16_values(rng, shape, scale=1.0, offset=None):
    x = rng.standard_normal(shape).astype(np.float32) * np.float32(scale)
    if offset is not None:
        x = x + offset
    # round to bf16 exactly as the inputs are stored (RN-even on the bit pattern)
    u = x.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


# ---------------------------------------------------------------- key mean --

@pytest.mark.parametrize("s_len", [1, 5, 31, 32, 33, 100, 257])
def test_key_mean_matches_exact_rational(s_len):
    rng = np.random.default_rng(s_len)
    k = _bf16_values(rng, (s_len, 6), scale=2.0, offset=np.float32(1.5))
    got = key_mean_fp64(k)
    for d in range(k.shape[1]):
        exact = sum((Fraction(float(v)) for v in k[:, d]), Fraction(0)) / s_len
        # fp64 sums of these values are exact, so the oracle's value is
        # fl32(fl64(T / S)); that equals fl32(T / S) unless the fp64 quotient
        # lands on a float32 midpoint, which these inputs avoid.
        assert got[d] == f32_round(exact), (d, got[d], float(exact))


def test_key_mean_matches_fsum_at_config_shapes():
    rng = np.random.default_rng(7)
    for s_len, off in [(256, 0.0), (1024, 3.0)]:
        k = _bf16_values(rng, (s_len, 128), offset=(rng.standard_normal(128) * off).astype(np.float32))
        got = key_mean_fp64(k)
        ref = np.array([np.float32(math.fsum(k[:, d].astype(np.float64)) / s_len) for d in range(128)])
        assert np.array_equal(got, ref)


def test_key_mean_order_within_chunk():
    # Reading: each 32-token chunk is summed left to right in fp64. With
    # 2^60, 1, -2^60 the 1 is absorbed (2^60 + 1 rounds to 2^60), so the chunk
    # sums to 0, not to the exact 1.
    k = np.zeros((32, 1), np.float32)
    k[0, 0], k[1, 0], k[2, 0] = 2.0 ** 60, 1.0, -(2.0 ** 60)
    assert key_mean_fp64(k)[0] == 0.0
    # Reordered so the small value comes first, the sum is exact: 1/32.
    k2 = np.zeros((32, 1), np.float32)
    k2[0, 0], k2[1, 0], k2[2, 0] = 1.0, 2.0 ** 60, -(2.0 ** 60)
    assert key_mean_fp64(k2)[0] == np.float32(0.0)  # 1 + 2^60 also absorbs the 1
    k3 = np.zeros((32, 1), np.float32)
    k3[0, 0], k3[1, 0], k3[2, 0] = 2.0 ** 60, -(2.0 ** 60), 1.0
    assert key_mean_fp64(k3)[0] == np.float32(1.0 / 32.0)


def test_key_mean_pairwise_tree_over_chunks():
    # Reading: chunk sums combine by a pairwise tree. Chunks hold 2^60, 1,
    # -2^60, 1 (one nonzero token each). Tree: (2^60 + 1) + (-2^60 + 1) =
    # 2^60 + (-2^60) = 0. A left-to-right pass would give ((2^60+1)-2^60)+1 = 1.
    k = np.zeros((128, 1), np.float32)
    k[0, 0], k[32, 0], k[64, 0], k[96, 0] = 2.0 ** 60, 1.0, -(2.0 ** 60), 1.0
    assert key_mean_fp64(k)[0] == 0.0
    # Three chunks pad to four with +0.0: (2^60 + 1) + (-2^60 + 0) = 0.
    k5 = np.zeros((96, 1), np.float32)
    k5[0, 0], k5[32, 0], k5[64, 0] = 2.0 ** 60, 1.0, -(2.0 ** 60)
    assert key_mean_fp64(k5)[0] == 0.0


def test_key_mean_of_negative_zeros_is_positive_zero():
    k = np.full((40, 2), -0.0, np.float32)
    m = key_mean_fp64(k)
    assert np.all(m == 0) and not np.any(np.signbit(m))


# ----------------------------------------------------------- int8 blocks --

def _int8_bruteforce(x):
    s_len, d = x.shape
    n_blk = -(-s_len // QK_BLOCK)
    codes = np.zeros((s_len, d), np.int8)
    scales = np.zeros(n_blk, np.float32)
    for t in range(n_blk):
        rows = range(t * QK_BLOCK, min((t + 1) * QK_BLOCK, s_len))
        amax = max(abs(Fraction(float(x[r, c]))) for r in rows for c in range(d))
        if amax == 0:
            continue
        s = f32_round(amax / INT8_MAX)
        scales[t] = s
        for r in rows:
            for c in range(d):
                q = f32_round(Fraction(float(x[r, c])) / Fraction(float(s)))
                codes[r, c] = max(-INT8_MAX, min(INT8_MAX, round_half_even(Fraction(float(q)))))
    return codes, scales


@pytest.mark.parametrize("s_len,seed", [(1, 0), (33, 1), (70, 2), (96, 3)])
def test_int8_blocks_bruteforce(s_len, seed):
    rng = np.random.default_rng(seed)
    # magnitudes spread over many binades, plus exact ties of x/s with .5
    x = _bf16_values(rng, (s_len, 8)) * np.float32(2.0) ** rng.integers(-20, 20, (s_len, 8)).astype(np.float32)
    got_c, got_s = quantize_int8_blocks(x)
    ref_c, ref_s = _int8_bruteforce(x)
    assert np.array_equal(got_s.view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(got_c, ref_c)


def test_int8_round_half_even_ties():
    # amax = 127 gives s = 1 exactly, so x/s = x and the .5 ties are visible.
    x = np.zeros((32, 4), np.float32)
    x[0] = [127.0, 0.5, 1.5, 2.5]
    x[1] = [-0.5, -1.5, -2.5, 126.5]
    c, s = quantize_int8_blocks(x)
    assert s[0] == 1.0
    assert c[0].tolist() == [127, 0, 2, 2]
    assert c[1].tolist() == [0, -2, -2, 126]


def test_int8_invariants_and_zero_blocks():
    rng = np.random.default_rng(11)
    x = _bf16_values(rng, (200, 128), scale=3.0)
    x[64:96] = 0.0           # an all-zero block
    c, s = quantize_int8_blocks(x)
    assert s.shape == (7,)
    assert s[2] == 0 and np.all(c[64:96] == 0)
    assert np.all(np.abs(c.astype(np.int32)) <= INT8_MAX)
    for t in range(7):
        if s[t] == 0:
            continue
        blk = slice(t * 32, min(t * 32 + 32, 200))
        assert np.abs(c[blk].astype(np.int32)).max() == INT8_MAX
        err = np.abs(c[blk].astype(np.float64) * s[t] - x[blk].astype(np.float64))
        assert err.max() <= 0.5 * s[t] * (1 + 1e-6)


# --------------------------------------------------------------- V channels --

def test_v_channels_bruteforce():
    rng = np.random.default_rng(21)
    v = _bf16_values(rng, (45, 6)) * np.float32(2.0) ** rng.integers(-6, 6, (45, 6)).astype(np.float32)
    v[:, 3] = 0.0
    got_c, got_s = quantize_v_channels(v)
    for d in range(6):
        amax = max(abs(Fraction(float(t))) for t in v[:, d])
        if amax == 0:
            assert got_s[d] == 0 and np.all(got_c[:, d] == 0)
            continue
        s = f32_round(amax / Fraction(448))
        assert got_s[d] == s
        for r in range(45):
            q = f32_round(Fraction(float(v[r, d])) / Fraction(float(s)))
            assert int(got_c[r, d]) == e4m3_round_bruteforce(float(q)), (r, d)


def test_v_channel_max_maps_to_448():
    rng = np.random.default_rng(22)
    v = _bf16_values(rng, (300, 128))
    c, s = quantize_v_channels(v)
    dec = e4m3_decode(c)
    for d in range(128):
        i = int(np.argmax(np.abs(v[:, d])))
        assert abs(float(dec[i, d])) == E4M3_MAX
    assert np.all(np.abs(dec) <= E4M3_MAX)
    # decoded codes times scale reproduce V to e4m3 precision: half a step,
    # i.e. 2^-4 relative in the normal range and 2^-10 * s below 2^-6 * s
    err = np.abs(dec.astype(np.float64) * s[None, :] - v)
    bound = np.maximum(2.0 ** -4 * np.abs(v), 2.0 ** -10 * s[None, :]) * (1 + 1e-5)
    assert np.all(err <= bound)


# ----------------------------------------------------------------- smooth_k --

def test_smooth_k_subtracts_mean_in_fp32():
    rng = np.random.default_rng(31)
    q = _bf16_values(rng, (64, 128))
    k = _bf16_values(rng, (64, 128), offset=(rng.standard_normal(128) * 3).astype(np.float32))
    v = _bf16_values(rng, (64, 128))
    on = quantize_head(q, k, v, smooth_k=True)
    off = quantize_head(q, k, v, smooth_k=False)
    assert np.array_equal(off["k_mean"], np.zeros(128, np.float32))
    kc, ks = quantize_int8_blocks((k - on["k_mean"][None, :]).astype(np.float32))
    assert np.array_equal(on["k_codes"], kc) and np.array_equal(on["k_scale"], ks)
    assert np.array_equal(on["q_codes"], off["q_codes"])
    assert np.array_equal(on["v_codes"], off["v_codes"])
    # the offset dominates K before smoothing, so the scales shrink after it
    assert on["k_scale"].max() < off["k_scale"].max()


def test_quantize_tensors_layouts_agree():
    rng = np.random.default_rng(41)
    b, s, h, d = 2, 100, 3, 128
    q = _bf16_values(rng, (b, s, h, d))
    k = _bf16_values(rng, (b, s, h, d))
    v = _bf16_values(rng, (b, s, h, d))
    nhd = quantize_tensors(q, k, v, "NHD", True)
    hnd = quantize_tensors(q.transpose(0, 2, 1, 3).copy(), k.transpose(0, 2, 1, 3).copy(),
                           v.transpose(0, 2, 1, 3).copy(), "HND", True)
    for key in nhd:
        assert np.array_equal(nhd[key], hnd[key]), key
    assert nhd["q_codes"].shape == (b, h, 128, d) and np.all(nhd["q_codes"][:, :, s:] == 0)
    assert nhd["vt_codes"].shape == (b, h, d, 128) and np.all(nhd["vt_codes"][:, :, :, s:] == 0)
    assert nhd["q_scale"].shape == (b, h, 4) and np.all(nhd["q_scale"][:, :, 4:] == 0)
