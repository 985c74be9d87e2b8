"""The causal mask and the log-sum-exp on the GPU (sage_attention_ex,
sage_sageattn_ex, sage_lse_smooth_k_term, and the SIMT cross-check) against
the oracle.

Outputs: max |gpu - emulation| <= 2e-2 and mean <= 2e-3 (bf16), cosine against
exact fp64 attention as for the unmasked path. Log-sum-exp: the GPU evaluates
the same online softmax in base 2 with ex2.approx and another fp32 summation
order; each row's m agrees to a few fp32 ulps of the logits (|logit| < 64 here)
and l to about 1e-6 relative, so |lse_gpu - lse_emulation| <= 2e-4 is a loose
bound; the smooth_k term adds an fp32 dot product of 128 terms (relative
error about 1e-6 of its magnitude).
"""

import math

import numpy as np
import pytest
import torch

from gpu_util import ATOL_MAX, ATOL_MEAN, COS_MIN, COS_SLACK, cosine, head_out, to_np
from oracle.tensors import attention_from_codes, exact_head, quantize_tensors
from quantized_attention_fp64_gb300 import (attention, attention_simt, device_error, lse_smooth_k_term, quantize,
                                            sageattn, sageattn_ex)
from quantized_attention_fp64_gb300.workloads import WORKLOADS, custom, make_qkv

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(128.0)
LSE_ATOL = 2e-4


def _check(out, lse, q, k, v, layout, ref, causal, heads, rows=None, lse_with_term=False):
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    s_len = qn.shape[1] if layout == "NHD" else qn.shape[2]
    errs, got_all, emu_all, ex_all = [], [], [], []
    for b, h in heads:
        emu, emu_lse = attention_from_codes(ref, s_len, SM, b, h, rows=rows, causal=causal, return_lse=True,
                                            q=qn if lse_with_term else None, layout=layout)
        ex = exact_head(qn, kn, vn, layout, SM, b, h, rows=rows, causal=causal)
        got = head_out(out, layout, b, h)
        got = got if rows is None else got[rows]
        errs.append(np.abs(got.astype(np.float64) - emu).ravel())
        got_all.append(got.ravel()), emu_all.append(emu.ravel()), ex_all.append(ex.ravel())
        if lse is not None:
            gl = lse[b, h] if rows is None else lse[b, h][rows]
            d = np.abs(gl.astype(np.float64) - emu_lse.astype(np.float64))
            assert d.max() <= LSE_ATOL, f"lse head {(b, h)}: max diff {d.max()}"
    err = np.concatenate(errs)
    assert err.max() <= ATOL_MAX and err.mean() <= ATOL_MEAN, (err.max(), err.mean())
    ex = np.concatenate(ex_all)
    cos, cos_emu = cosine(np.concatenate(got_all), ex), cosine(np.concatenate(emu_all), ex)
    assert cos >= min(COS_MIN, cos_emu - COS_SLACK), (cos, cos_emu)


@pytest.mark.parametrize("s_len", [1, 33, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_attention_ex_matches_oracle(sage_lib, s_len, causal):
    w = custom(1, 2, s_len, seed_index=800 + s_len, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", True)
    out, lse = attention(qz, SM, is_causal=causal, return_lse=True)
    torch.cuda.synchronize()
    assert device_error() == 0
    ref = quantize_tensors(to_np(q), to_np(k), to_np(v), "NHD", True)
    _check(to_np(out), lse.cpu().numpy(), q, k, v, "NHD", ref, causal, [(0, 0), (0, 1)])


@pytest.mark.parametrize("s_len", [2048, 2200])
def test_lse_with_correction_warpgroup(sage_lib, s_len):
    # unmasked rows of 16 key tiles or more run the kernel with the correction
    # warpgroup; the log-sum-exp comes from the same softmax state
    w = custom(1, 2, s_len, seed_index=850 + s_len, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", True)
    out, lse = attention(qz, SM, is_causal=False, return_lse=True)
    torch.cuda.synchronize()
    assert device_error() == 0
    ref = quantize_tensors(to_np(q), to_np(k), to_np(v), "NHD", True)
    rows = np.unique(np.concatenate([np.arange(0, s_len, 29), np.arange(s_len - 3, s_len)]))
    _check(to_np(out), lse.cpu().numpy(), q, k, v, "NHD", ref, False, [(0, 0), (0, 1)], rows=rows)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_sageattn_ex_causal_lse_with_smooth_k_term(sage_lib, layout):
    w = WORKLOADS["B2_H8_S1024"]
    q, k, v = make_qkv(w, "cuda", layout)
    out, lse = sageattn_ex(q, k, v, tensor_layout=layout, is_causal=True, sm_scale=SM, return_lse=True)
    torch.cuda.synchronize()
    assert device_error() == 0
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    ref = quantize_tensors(qn, kn, vn, layout, True)
    heads = [(0, 0), (1, 3), (1, 7)]
    _check(to_np(out), lse.cpu().numpy(), q, k, v, layout, ref, True, heads, lse_with_term=True)
    # with the key-mean term the GPU's lse tracks the exact one closely
    for b, h in heads:
        _, ex_lse = exact_head(qn, kn, vn, layout, SM, b, h, causal=True, return_lse=True)
        assert np.abs(lse[b, h].cpu().numpy() - ex_lse).max() <= 0.05


def test_lse_smooth_k_term_entry(sage_lib):
    w = custom(2, 3, 777, seed_index=850, k_offset_std=3.0)
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", True)
    _, lse = attention(qz, SM, return_lse=True)
    base = lse.clone()
    lse_smooth_k_term(q, qz, lse, SM)
    torch.cuda.synchronize()
    term = SM * torch.einsum("bshd,bhd->bhs", q.double(), qz.k_mean.double())
    assert torch.allclose((lse - base).double(), term, rtol=1e-5, atol=1e-4)


def test_non_causal_ex_equals_plain_attention(sage_lib):
    w = custom(2, 4, 777, seed_index=860, k_offset_std=1.0)
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", True)
    a = attention(qz, SM)
    b, _ = attention(qz, SM, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("causal", [True, False])
def test_tc_and_simt_agree_with_mask_and_lse(sage_lib, causal):
    w = custom(2, 3, 650, seed_index=870, k_offset_std=1.5)
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", True)
    a, la = attention(qz, SM, is_causal=causal, return_lse=True)
    b, lb = attention_simt(qz, SM, is_causal=causal, return_lse=True)
    torch.cuda.synchronize()
    d = (a.float() - b.float()).abs()
    assert d.max().item() <= ATOL_MAX and d.mean().item() <= ATOL_MEAN
    assert (la - lb).abs().max().item() <= LSE_ATOL


def test_causal_video_size_sampled_rows(sage_lib):
    # the bench workload with the causal mask: sampled rows of three heads,
    # including the first and last rows of the sequence
    w = WORKLOADS["B1_H28_S16384"]
    q, k, v = make_qkv(w, "cuda")
    out, lse = sageattn_ex(q, k, v, is_causal=True, sm_scale=SM, return_lse=True)
    torch.cuda.synchronize()
    assert device_error() == 0
    rows = np.concatenate([[0, 1, 127, 128, 16383], np.random.default_rng(4).choice(16384, 60, replace=False)])
    rows = np.unique(rows)
    heads = [(0, 0), (0, 13), (0, 27)]
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    ref = quantize_tensors(qn, kn, vn, "NHD", True, heads=heads)
    _check(to_np(out), lse.cpu().numpy(), q, k, v, "NHD", ref, True, heads, rows=rows, lse_with_term=True)


def test_plain_sageattn_still_rejects_causal_and_lse(sage_lib):
    from quantized_attention_fp64_gb300 import SageError
    q = torch.zeros(1, 64, 2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(SageError):
        sageattn(q, q, q, is_causal=True)
    with pytest.raises(SageError):
        sageattn(q, q, q, return_lse=True)
