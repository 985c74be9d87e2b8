"""The tcgen05 attention kernel (sage_attention / sage_sageattn) against the
oracle: max/mean abs error against the quantized emulation, cosine against
exact fp64 attention, and agreement with the independent SIMT kernel."""

import math

import numpy as np
import pytest
import torch

from gpu_util import check_attention, to_np
from oracle.tensors import quantize_tensors
from quantized_attention_fp64_gb300 import attention, attention_simt, device_error, quantize, sageattn
from quantized_attention_fp64_gb300.workloads import WORKLOADS, custom, make_qkv

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(128.0)


def _tc_vs_oracle(w, layout="NHD", heads=None, rows=None):
    q, k, v = make_qkv(w, "cuda", layout)
    qz = quantize(q, k, v, layout, w.smooth_k)
    out = attention(qz, SM, tensor_layout=layout)
    torch.cuda.synchronize()
    assert device_error() == 0
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    heads = heads or [(b, h) for b in range(w.B) for h in range(w.H)]
    ref = quantize_tensors(qn, kn, vn, layout, w.smooth_k, heads=heads)
    return check_attention(to_np(out), qn, kn, vn, layout, ref, SM, heads, rows=rows), (qz, out)


@pytest.mark.parametrize("w", [WORKLOADS["B1_H2_S256"], WORKLOADS["B2_H8_S1024"],
                               custom(1, 2, 128, seed_index=401), custom(1, 3, 384, seed_index=402)])
def test_tc_matches_oracle(sage_lib, w):
    _tc_vs_oracle(w)


@pytest.mark.parametrize("s_len", [1, 33, 127, 129, 200, 1000, 2047, 2048, 2200, 4097])
def test_tc_ragged_lengths(sage_lib, s_len):
    # from 16 key tiles (S > 1920) the kernel runs with its correction
    # warpgroup; below, the softmax warps rescale O themselves
    _tc_vs_oracle(custom(1, 2, s_len, seed_index=500 + s_len, k_offset_std=2.0))


@pytest.mark.parametrize("B,H,S", [(2, 40, 2200), (1, 20, 3001)])
def test_tc_tile_pairs_with_correction_warpgroup(sage_lib, B, H, S):
    # enough heads for two query tiles per unit, long enough rows for the
    # correction warpgroup, a ragged last key tile; sampled heads
    _tc_vs_oracle(custom(B, H, S, seed_index=510 + H, k_offset_std=1.5), heads=[(0, 0), (B - 1, H - 1), (0, H // 2)])


def test_tc_hnd_layout(sage_lib):
    _tc_vs_oracle(WORKLOADS["B2_H8_S1024"], layout="HND")


def test_tc_agrees_with_simt(sage_lib):
    w = custom(2, 4, 777, seed_index=601, k_offset_std=1.0)
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", True)
    a = attention(qz, SM)
    b = attention_simt(qz, SM)
    torch.cuda.synchronize()
    d = (a.float() - b.float()).abs()
    assert d.max().item() <= 2e-2 and d.mean().item() <= 2e-3


def test_tc_image_size_sampled_heads(sage_lib):
    _tc_vs_oracle(WORKLOADS["B1_H28_S4096"], heads=[(0, 0), (0, 11), (0, 27)])


def test_tc_video_size_sampled_rows(sage_lib):
    # the bench configuration at full size; the oracle checks sampled rows of
    # three heads (the emulation of a row does not depend on the other rows)
    rows = np.sort(np.random.default_rng(3).choice(16384, 160, replace=False))
    _tc_vs_oracle(WORKLOADS["B1_H28_S16384"], heads=[(0, 0), (0, 14), (0, 27)], rows=rows)


def test_sageattn_entry(sage_lib):
    w = custom(1, 2, 300, seed_index=701, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda")
    out = sageattn(q, k, v, tensor_layout="NHD", is_causal=False, sm_scale=None, return_lse=False)
    torch.cuda.synchronize()
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    ref = quantize_tensors(qn, kn, vn, "NHD", True)
    check_attention(to_np(out), qn, kn, vn, "NHD", ref, SM, [(0, 0), (0, 1)])


@pytest.mark.parametrize("kw", [dict(is_causal=True), dict(return_lse=True)])
def test_sageattn_rejects_on_gpu(sage_lib, kw):
    from quantized_attention_fp64_gb300 import SageError
    q = torch.zeros(1, 64, 2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(SageError):
        sageattn(q, q, q, **kw)
    with pytest.raises(SageError):
        sageattn(q.float(), q.float(), q.float())
    with pytest.raises(SageError):
        sageattn(q[..., :64].contiguous(), q[..., :64].contiguous(), q[..., :64].contiguous())
    with pytest.raises(SageError):
        sageattn(q, q[:, :32].contiguous(), q)
