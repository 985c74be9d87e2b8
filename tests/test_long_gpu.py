"""The longest workloads on the GPU against the oracle, on sampled heads and
query rows: B1 H28 S131072 and B1 H80 S131072, whose bf16 tensors (2.7 GB
each at 80 heads) put element offsets past 2^31 bytes.

The kernels run on the full tensors; the oracle runs on the sampled heads
only, sliced out on the GPU before the copy to the host (heads are
independent, so the oracle of a slice is the oracle of those heads). The
prologue must match bit for bit on those heads; attention meets the usual
bounds (max |gpu - emulation| <= 2e-2, mean <= 2e-3, cosine against exact
fp64 attention) on the sampled rows, unmasked and causal.
"""

import math

import numpy as np
import pytest
import torch

from gpu_util import ATOL_MAX, ATOL_MEAN, COS_MIN, COS_SLACK, assert_bundles_equal, cosine, to_np
from oracle.tensors import attention_from_codes, exact_head, quantize_tensors
from quantized_attention_fp64_gb300 import attention, device_error, quantize
from quantized_attention_fp64_gb300.workloads import WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(128.0)


def _bundle_heads(qz, hs):
    """The bundle's arrays for heads hs of batch 0, as a 1-batch bundle."""
    def take(t):
        return t[0:1, hs].contiguous().cpu().numpy()
    return dict(q_codes=take(qz.q_codes), k_codes=take(qz.k_codes), vt_codes=take(qz.vt_codes),
                q_scale=take(qz.q_scale), k_scale=take(qz.k_scale), v_scale=take(qz.v_scale),
                k_mean=take(qz.k_mean))


def _attention_close(out_s, q_s, k_s, v_s, ref, rows, causal):
    """out_s, q_s, k_s, v_s: [1, S, n, 128] numpy slices; ref: the oracle
    bundle of the slice."""
    s_len = q_s.shape[1]
    errs, got_all, emu_all, ex_all = [], [], [], []
    for h in range(q_s.shape[2]):
        emu = attention_from_codes(ref, s_len, SM, 0, h, rows=rows, causal=causal)
        ex = exact_head(q_s, k_s, v_s, "NHD", SM, 0, h, rows=rows, causal=causal)
        got = out_s[0, rows, h, :].astype(np.float64)
        errs.append(np.abs(got - emu).ravel())
        got_all.append(got.ravel()), emu_all.append(emu.ravel()), ex_all.append(ex.ravel())
    err = np.concatenate(errs)
    assert err.max() <= ATOL_MAX and err.mean() <= ATOL_MEAN, (err.max(), err.mean())
    ex = np.concatenate(ex_all)
    cos, cos_emu = cosine(np.concatenate(got_all), ex), cosine(np.concatenate(emu_all), ex)
    assert cos >= min(COS_MIN, cos_emu - COS_SLACK), (cos, cos_emu)


@pytest.mark.parametrize("name,heads", [("B1_H28_S131072", [0, 27]), ("B1_H80_S131072", [0, 79])])
def test_longest_sequences_sampled(sage_lib, name, heads):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", w.smooth_k)
    out = attention(qz, SM)
    out_c = attention(qz, SM, is_causal=True)
    torch.cuda.synchronize()
    assert device_error() == 0
    hs = torch.tensor(heads, device="cuda")
    q_s, k_s, v_s = (to_np(t.index_select(2, hs)) for t in (q, k, v))
    ref = quantize_tensors(q_s, k_s, v_s, "NHD", w.smooth_k)
    assert_bundles_equal(_bundle_heads(qz, hs), ref)
    # rows across the sequence, the last ones included (offsets near the end
    # of the tensors)
    rows = np.unique(np.concatenate([np.random.default_rng(17).choice(w.S, 20, replace=False),
                                     np.arange(w.S - 4, w.S)]))
    _attention_close(to_np(out.index_select(2, hs)), q_s, k_s, v_s, ref, rows, causal=False)
    _attention_close(to_np(out_c.index_select(2, hs)), q_s, k_s, v_s, ref, rows, causal=True)
