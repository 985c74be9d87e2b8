"""The pins catch plausible mistakes in the oracle.

Each test plants one mistake (a wrong rounding mode, a wrong constant, a
dropped or misplaced term, a transposed operand, an off-by-one mask) in a
copy of an oracle function, on the CPU, and checks that the pin written
against that function now fails. The mistakes live only inside these tests
(monkeypatched for the duration of one test); the oracle itself is untouched.
"""

import numpy as np
import pytest

import oracle.sage_oracle as so
import test_oracle_attention as A
import test_oracle_causal_lse as C
import test_oracle_formats as F
import test_oracle_prologue as P

ORIG_MEAN = so.key_mean_fp64
ORIG_EXACT = so.attention_exact
ORIG_EMU = so.attention_emulated


def _fails(pin, *args):
    with pytest.raises(AssertionError):
        with np.errstate(all="ignore"):
            pin(*args)


# ------------------------------------------------------------- INT8 blocks --

def _int8_with(x32, divisor=127.0, half_up=False):
    x32 = np.asarray(x32, np.float32)
    s_len = x32.shape[0]
    n_blk = -(-s_len // 32)
    codes = np.zeros(x32.shape, np.int8)
    scales = np.zeros(n_blk, np.float32)
    for t in range(n_blk):
        blk = slice(t * 32, min(t * 32 + 32, s_len))
        amax = np.float32(np.abs(x32[blk]).max())
        if amax == 0:
            continue
        s = np.float32(amax / np.float32(divisor))
        q = (x32[blk] / s).astype(np.float32)
        r = np.sign(q) * np.floor(np.abs(q) + 0.5) if half_up else np.rint(q)
        codes[blk] = np.clip(r, -127, 127).astype(np.int8)
        scales[t] = s
    return codes, scales


def test_int8_ties_rounded_half_away_from_zero_is_caught(monkeypatch):
    monkeypatch.setattr(P, "quantize_int8_blocks", lambda x: _int8_with(x, half_up=True))
    _fails(P.test_int8_round_half_even_ties)


def test_int8_scale_amax_over_128_is_caught(monkeypatch):
    monkeypatch.setattr(P, "quantize_int8_blocks", lambda x: _int8_with(x, divisor=128.0))
    _fails(P.test_int8_blocks_bruteforce, 33, 1)


def test_the_planted_int8_copy_is_faithful_without_a_mistake(monkeypatch):
    # guards the two tests above: the copy itself passes the pins
    monkeypatch.setattr(P, "quantize_int8_blocks", lambda x: _int8_with(x))
    P.test_int8_round_half_even_ties()
    P.test_int8_blocks_bruteforce(33, 1)


# ---------------------------------------------------------------- key mean --

def _mean_fp32_accumulation(k32):
    k32 = np.asarray(k32, np.float32)
    acc = np.zeros(k32.shape[1], np.float32)
    for s in range(k32.shape[0]):
        acc = (acc + k32[s]).astype(np.float32)
    return (acc.astype(np.float64) / k32.shape[0]).astype(np.float32)


def _mean_chunks_left_to_right(k32):
    k32 = np.asarray(k32, np.float32)
    s_len = k32.shape[0]
    total = np.zeros(k32.shape[1], np.float64)
    for c in range(0, s_len, 32):
        part = np.zeros(k32.shape[1], np.float64)
        for s in range(c, min(c + 32, s_len)):
            part = part + k32[s].astype(np.float64)
        total = total + part
    return (total / s_len).astype(np.float32)


def test_key_mean_summed_in_fp32_is_caught(monkeypatch):
    monkeypatch.setattr(P, "key_mean_fp64", _mean_fp32_accumulation)
    _fails(P.test_key_mean_matches_fsum_at_config_shapes)


def test_key_mean_chunks_joined_left_to_right_is_caught(monkeypatch):
    monkeypatch.setattr(P, "key_mean_fp64", _mean_chunks_left_to_right)
    _fails(P.test_key_mean_pairwise_tree_over_chunks)


def test_smooth_k_adding_the_mean_is_caught(monkeypatch):
    # quantize_head looks the key mean up in the oracle module: a sign error
    # there makes it quantize k + mean
    monkeypatch.setattr(so, "key_mean_fp64", lambda k: -ORIG_MEAN(k))
    _fails(P.test_smooth_k_subtracts_mean_in_fp32)


# --------------------------------------------------------------- V channels --

def test_v_scale_amax_over_447_is_caught(monkeypatch):
    def v_447(v32):
        v32 = np.asarray(v32, np.float32)
        scales = (np.abs(v32).max(axis=0) / np.float32(447.0)).astype(np.float32)
        codes = np.zeros(v32.shape, np.uint8)
        live = scales > 0
        codes[:, live] = so.e4m3_encode((v32[:, live] / scales[live][None, :]).astype(np.float32))
        return codes, scales
    monkeypatch.setattr(P, "quantize_v_channels", v_447)
    _fails(P.test_v_channels_bruteforce)


# ------------------------------------------------------------------ e4m3 --

def test_e4m3_encode_truncating_is_caught(monkeypatch):
    vals = so.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)  # 0 .. 448, increasing

    def truncate(x):
        x = np.asarray(x, np.float32).astype(np.float64)
        mag = np.minimum(np.abs(x), 448.0)
        code = np.searchsorted(vals, mag, side="right") - 1
        code = np.where(np.isnan(x), 0x7F, code)
        return (code | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)

    monkeypatch.setattr(F, "e4m3_encode", truncate)
    _fails(F.test_e4m3_encode_hand_cases)


# -------------------------------------------------------- exact attention --

def test_exact_attention_with_q_and_k_swapped_is_caught(monkeypatch):
    monkeypatch.setattr(A, "attention_exact", lambda q, k, v, sm, **kw: ORIG_EXACT(k, q, v, sm, **kw))
    _fails(A.test_exact_matches_python_bruteforce, 3, 4)


def test_exact_attention_without_sm_scale_is_caught(monkeypatch):
    monkeypatch.setattr(A, "attention_exact", lambda q, k, v, sm, **kw: ORIG_EXACT(q, k, v, 1.0, **kw))
    _fails(A.test_exact_matches_python_bruteforce, 8, 5)


# --------------------------------------------------------------- emulation --

def test_emulation_without_v_scales_is_caught(monkeypatch):
    def no_v_scale(qc, kc, vv, sq, sk, sv, sm, **kw):
        return ORIG_EMU(qc, kc, vv, sq, sk, np.full_like(np.asarray(sv), 1.0 / 448.0), sm, **kw)
    monkeypatch.setattr(A, "attention_emulated", no_v_scale)
    _fails(A.test_emulation_scale_indexing)


def test_emulation_with_q_and_k_scales_swapped_is_caught(monkeypatch):
    monkeypatch.setattr(A, "attention_emulated",
                        lambda qc, kc, vv, sq, sk, sv, sm, **kw: ORIG_EMU(qc, kc, vv, sk, sq, sv, sm, **kw))
    _fails(A.test_emulation_scale_indexing)


def test_causal_mask_off_by_one_is_caught(monkeypatch):
    def strict(rows, j0, j1, causal):
        if not causal:
            return None
        return np.arange(j0, j1)[None, :] < np.asarray(rows)[:, None]
    monkeypatch.setattr(so, "_visible", strict)
    _fails(C.test_emulation_causal_reduces_to_exact_without_quantization, 100)


def test_lse_without_the_smooth_k_term_is_caught(monkeypatch):
    monkeypatch.setattr(C, "smooth_k_lse_term", lambda q, mean, sm, rows=None: np.zeros(np.asarray(q).shape[0]))
    _fails(C.test_emulated_lse_needs_and_gets_the_smooth_k_term, False)


def test_p_stored_without_its_448_scale_is_caught(monkeypatch):
    # the emulation reads the P scale from the oracle module at call time
    monkeypatch.setattr(so, "P_SCALE", 1.0)
    _fails(A.test_emulation_single_tile_closed_form)


def _emulated_plain(qc, kc, vv, sq, sk, sv, sm, quantize_p=True, return_fp32=False, drop_alpha=False):
    """A plain copy of the emulation's loop (unmasked, all rows), with an
    optional planted mistake: the accumulator not rescaled by alpha."""
    f32, f64 = np.float32, np.float64
    qc, kc = np.asarray(qc), np.asarray(kc)
    s_len, d = kc.shape
    sq = np.asarray(sq, f32)[np.arange(qc.shape[0]) // 32]
    sk, sv, vv, scale = np.asarray(sk, f32), np.asarray(sv, f32), np.asarray(vv, f32), f32(sm)
    m = np.full(qc.shape[0], -np.inf, f32)
    l = np.zeros(qc.shape[0], f32)
    acc = np.zeros((qc.shape[0], d), f32)
    for j0 in range(0, s_len, 128):
        j1 = min(j0 + 128, s_len)
        s_ij = qc.astype(f64) @ kc[j0:j1].astype(f64).T
        c = ((sq[:, None] * sk[np.arange(j0, j1) // 32][None, :]).astype(f32) * scale).astype(f32)
        logit = (s_ij.astype(f32) * c).astype(f32)
        m_new = np.maximum(m, logit.max(axis=1))
        alpha = np.exp((m - m_new).astype(f64)).astype(f32)
        alpha = np.where(m == m_new, f32(1.0), alpha).astype(f32)
        p = np.exp((logit - m_new[:, None]).astype(f32).astype(f64)).astype(f32)
        l = (alpha * l + p.astype(f64).sum(axis=1).astype(f32)).astype(f32)
        p448 = (f32(448.0) * p).astype(f32)
        p_used = so.e4m3_decode(so.e4m3_encode(p448)) if quantize_p else p448
        pv = (p_used.astype(f64) @ vv[j0:j1].astype(f64)).astype(f32)
        acc = ((acc if drop_alpha else alpha[:, None] * acc) + pv).astype(f32)
        m = m_new
    out = ((((acc / l[:, None]).astype(f32)) * sv[None, :]).astype(f32) / f32(448.0)).astype(f32)
    return out if return_fp32 else so.bf16_round(out)


def test_accumulator_not_rescaled_by_alpha_is_caught(monkeypatch):
    monkeypatch.setattr(A, "attention_emulated",
                        lambda *a, **kw: _emulated_plain(*a, drop_alpha=True, **kw))
    _fails(A.test_emulation_reduces_to_exact_without_quantization, 300)


def test_the_planted_emulation_copy_is_faithful_without_a_mistake(monkeypatch):
    monkeypatch.setattr(A, "attention_emulated", lambda *a, **kw: _emulated_plain(*a, **kw))
    A.test_emulation_reduces_to_exact_without_quantization(300)
    A.test_emulation_scale_indexing()
