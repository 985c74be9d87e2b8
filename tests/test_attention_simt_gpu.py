"""The SIMT cross-check kernel against the oracle's emulation and exact attention."""

import math

import pytest
import torch

from gpu_util import check_attention, to_np
from oracle.tensors import quantize_tensors
from quantized_attention_fp64_gb300 import attention_simt, quantize
from quantized_attention_fp64_gb300.workloads import WORKLOADS, custom, make_qkv

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(128.0)


@pytest.mark.parametrize("w", [WORKLOADS["B1_H2_S256"], WORKLOADS["B2_H8_S1024"],
                               custom(1, 2, 1, seed_index=301), custom(1, 2, 33, seed_index=302),
                               custom(1, 2, 1000, seed_index=303, k_offset_std=2.0)])
def test_simt_matches_oracle(sage_lib, w):
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", w.smooth_k)
    out = attention_simt(qz, SM)
    torch.cuda.synchronize()
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    ref = quantize_tensors(qn, kn, vn, "NHD", w.smooth_k)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    check_attention(to_np(out), qn, kn, vn, "NHD", ref, SM, heads)
