"""Pins for the oracle's attention: exact fp64 attention and the emulation.

References: pure-Python brute force (math.exp / math.fsum) on tiny inputs,
closed forms (S = 1, Q = 0, V = const), the smooth_k invariance that the
method relies on, reduction of the emulation to exact attention when every
quantization is the identity, and the accuracy level the pages report.
"""

import math

import numpy as np
import pytest

from oracle import (attention_emulated, attention_exact, e4m3_decode, e4m3_encode, quantize_head)

SM = np.float32(1.0 / math.sqrt(128.0))


def _round_bf16(x):
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(np.float32)


def _bf16(rng, shape, scale=1.0):
    return _round_bf16(rng.standard_normal(shape) * scale)


def _cos(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


# ------------------------------------------------------------ exact attention --

@pytest.mark.parametrize("s_len,d", [(1, 4), (3, 4), (8, 5)])
def test_exact_matches_python_bruteforce(s_len, d):
    rng = np.random.default_rng(s_len * 10 + d)
    q, k, v = (_bf16(rng, (s_len, d)) for _ in range(3))
    sm = float(np.float32(0.37))  # sm_scale crosses the C ABI as a float32
    got = attention_exact(q, k, v, sm)
    for i in range(s_len):
        logits = [sm * math.fsum(float(q[i, c]) * float(k[j, c]) for c in range(d)) for j in range(s_len)]
        mx = max(logits)
        w = [math.exp(t - mx) for t in logits]
        z = math.fsum(w)
        for c in range(d):
            ref = math.fsum(w[j] * float(v[j, c]) for j in range(s_len)) / z
            assert abs(got[i, c] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_exact_closed_forms():
    rng = np.random.default_rng(5)
    q, k, v = (_bf16(rng, (300, 128)) for _ in range(3))
    # S = 1: the only key gets weight 1
    assert np.allclose(attention_exact(q[:1], k[:1], v[:1], SM), v[:1], rtol=0, atol=1e-15)
    # V constant: every output equals that constant (rows of softmax sum to 1)
    ones = np.ones_like(v)
    assert np.abs(attention_exact(q, k, ones, SM) - 1.0).max() <= 1e-12
    # Q = 0: uniform weights, the output is the mean of V
    out = attention_exact(np.zeros_like(q), k, v, SM)
    assert np.abs(out - v.astype(np.float64).mean(axis=0)[None, :]).max() <= 1e-12
    # one dominant key: the output approaches that key's value
    k2 = k.copy()
    k2[17] = q[0] * np.float32(64.0)
    out = attention_exact(q[:1], k2, v, SM)
    assert np.abs(out[0] - v[17]).max() <= 1e-6


def test_exact_smooth_k_invariance():
    # A per-channel key shift adds q.mu to every logit of a row, which the
    # softmax cancels. Values on a 1/16 grid keep k - mu exact in float32.
    rng = np.random.default_rng(6)
    q = (rng.integers(-32, 32, (200, 128)) / 16).astype(np.float32)
    k = (rng.integers(-32, 32, (200, 128)) / 16).astype(np.float32)
    v = _bf16(rng, (200, 128))
    mu = (rng.integers(-48, 48, 128) / 16).astype(np.float32)
    a = attention_exact(q, k, v, SM)
    b = attention_exact(q, (k - mu[None, :]).astype(np.float32), v, SM)
    assert np.abs(a - b).max() <= 1e-12


# ----------------------------------------------------------------- emulation --

@pytest.mark.parametrize("s_len", [1, 100, 128, 129, 300])
def test_emulation_reduces_to_exact_without_quantization(s_len):
    # All codes are the values themselves, all scales 1, P kept in fp32: the
    # online softmax over 128-key tiles must reproduce exact attention.
    rng = np.random.default_rng(s_len)
    q, k, v = (_bf16(rng, (s_len, 128), 1.5) for _ in range(3))
    nb = -(-s_len // 32)
    got = attention_emulated(q, k, v, np.ones(nb, np.float32), np.ones(nb, np.float32),
                             np.ones(128, np.float32), SM, quantize_p=False, return_fp32=True)
    ref = attention_exact(q, k, v, SM)
    assert np.abs(got - ref).max() <= 2e-5 * np.abs(ref).max()


def test_emulation_scale_indexing():
    # Integer codes with different scales per 32-token block (Q and K) and per
    # channel (V): without P quantization the result must equal exact
    # attention of the dequantized tensors. A swapped or shifted scale index
    # breaks this.
    rng = np.random.default_rng(8)
    s_len = 230
    nb = -(-s_len // 32)
    qc = rng.integers(-127, 128, (s_len, 128)).astype(np.int8)
    kc = rng.integers(-127, 128, (s_len, 128)).astype(np.int8)
    sq = (rng.uniform(0.5, 2.0, nb) / 127).astype(np.float32)
    sk = (rng.uniform(0.5, 2.0, nb) / 127).astype(np.float32)
    vv = e4m3_decode(rng.integers(0, 0x7E, (s_len, 128)).astype(np.uint8) | (rng.integers(0, 2, (s_len, 128)) << 7).astype(np.uint8))
    sv = rng.uniform(0.1, 3.0, 128).astype(np.float32) / np.float32(448)
    got = attention_emulated(qc, kc, vv, sq, sk, sv, SM, quantize_p=False, return_fp32=True)
    qd = qc.astype(np.float64) * np.repeat(sq, 32)[:s_len, None]
    kd = kc.astype(np.float64) * np.repeat(sk, 32)[:s_len, None]
    vd = vv.astype(np.float64) * sv[None, :]
    logits = qd @ kd.T * float(SM)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    ref = (p @ vd) / p.sum(axis=1, keepdims=True)
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()


def test_emulation_single_tile_closed_form():
    # With one key tile the online softmax is a single step with the row's
    # global maximum: O = sum_j dec(e4m3(448 p_j)) v_j / sum_j p_j * s_v / 448,
    # the row sum taken over the unquantized p.
    rng = np.random.default_rng(9)
    s_len = 96
    qc = rng.integers(-127, 128, (s_len, 128)).astype(np.int8)
    kc = rng.integers(-127, 128, (s_len, 128)).astype(np.int8)
    sq = np.full(3, 0.02, np.float32)
    sk = np.full(3, 0.03, np.float32)
    vv = e4m3_decode(rng.integers(0, 0x7E, (s_len, 128)).astype(np.uint8))
    sv = np.full(128, 0.005, np.float32)
    got = attention_emulated(qc, kc, vv, sq, sk, sv, SM, return_fp32=True)
    logit = (qc.astype(np.float64) @ kc.astype(np.float64).T) * (0.02 * 0.03 * float(SM))
    p = np.exp(logit - logit.max(axis=1, keepdims=True))
    pt = e4m3_decode(e4m3_encode((448.0 * p).astype(np.float32))).astype(np.float64)
    ref = (pt @ vv.astype(np.float64)) / p.sum(axis=1, keepdims=True) * 0.005 / 448.0
    assert np.abs(got - ref).max() <= 1e-3 * np.abs(ref).max()
    # and P quantization is visible: without it the result moves
    plain = attention_emulated(qc, kc, vv, sq, sk, sv, SM, quantize_p=False, return_fp32=True)
    assert np.abs(plain - got).max() > 1e-4 * np.abs(ref).max()


def test_emulation_rows_subset_matches_full():
    rng = np.random.default_rng(10)
    q, k, v = (_bf16(rng, (333, 128)) for _ in range(3))
    r = quantize_head(q, k, v, smooth_k=False)
    vv = e4m3_decode(r["v_codes"])
    full = attention_emulated(r["q_codes"], r["k_codes"], vv, r["q_scale"], r["k_scale"], r["v_scale"], SM)
    rows = np.array([0, 5, 31, 32, 200, 332])
    sub = attention_emulated(r["q_codes"], r["k_codes"], vv, r["q_scale"], r["k_scale"], r["v_scale"], SM, rows=rows)
    assert np.array_equal(full[rows], sub)


@pytest.mark.parametrize("s_len,off,smooth", [(256, 0.0, False), (1024, 3.0, True), (1000, 2.0, True)])
def test_emulation_accuracy_vs_exact(s_len, off, smooth):
    # The pages report cosine 0.9992 against SDPA; the method must reach 0.999.
    rng = np.random.default_rng(s_len)
    q, v = _bf16(rng, (s_len, 128)), _bf16(rng, (s_len, 128))
    k = _round_bf16(rng.standard_normal((s_len, 128)) + rng.standard_normal(128)[None, :] * off)
    r = quantize_head(q, k, v, smooth_k=smooth)
    emu = attention_emulated(r["q_codes"], r["k_codes"], e4m3_decode(r["v_codes"]),
                             r["q_scale"], r["k_scale"], r["v_scale"], SM)
    ref = attention_exact(q, k, v, SM)
    assert _cos(emu, ref) >= 0.999


def test_smooth_k_does_not_hurt_with_key_offsets():
    rng = np.random.default_rng(12)
    s_len = 1024
    q, v = _bf16(rng, (s_len, 128)), _bf16(rng, (s_len, 128))
    k = _round_bf16(rng.standard_normal((s_len, 128)) + 3.0 * rng.standard_normal(128)[None, :])
    ref = attention_exact(q, k, v, SM)
    cos = {}
    for smooth in (False, True):
        r = quantize_head(q, k, v, smooth_k=smooth)
        emu = attention_emulated(r["q_codes"], r["k_codes"], e4m3_decode(r["v_codes"]),
                                 r["q_scale"], r["k_scale"], r["v_scale"], SM)
        cos[smooth] = _cos(emu, ref)
    assert cos[True] >= cos[False]
