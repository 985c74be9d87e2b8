"""Head dimension 64 on the GPU against the oracle: the prologue's codes,
scales and key means bit for bit, and attention (unmasked and causal, with
the log-sum-exp) within the output tolerances, through the bundle entries and
sage_sageattn_ex. The pages' sageattn entry itself keeps rejecting a head
dimension other than 128."""

import ctypes
import math

import numpy as np
import pytest
import torch

from gpu_util import assert_bundles_equal, bundle_np, check_attention, to_np
from oracle.tensors import attention_from_codes, quantize_tensors
from quantized_attention_fp64_gb300 import (SageError, attention, device_error, quantize, sageattn, sageattn_ex)
from quantized_attention_fp64_gb300 import _lib
from quantized_attention_fp64_gb300.api import _bf16_tensor, _stream, alloc_bundle
from quantized_attention_fp64_gb300.workloads import WORKLOADS, custom, make_qkv

pytestmark = pytest.mark.gpu
SM64 = 1.0 / math.sqrt(64.0)


def _prologue(q, k, v, layout, smooth, heads=None):
    qz = quantize(q, k, v, layout, smooth)
    torch.cuda.synchronize()
    assert qz.D == 64
    ref = quantize_tensors(to_np(q), to_np(k), to_np(v), layout, smooth, heads=heads)
    assert_bundles_equal(bundle_np(qz), ref, heads=heads)
    return qz


@pytest.mark.parametrize("s_len", [1, 31, 33, 129, 255, 1000, 1025, 1300])
@pytest.mark.parametrize("smooth", [True, False])
def test_prologue_d64_ragged(sage_lib, s_len, smooth):
    # 3 heads: the prologue runs head pairs, the second pair missing its
    # second head; up to 1024 tokens the cluster kernel, beyond the persistent one
    w = custom(2, 3, s_len, seed_index=1100 + s_len, k_offset_std=2.0, D=64)
    q, k, v = make_qkv(w, "cuda")
    _prologue(q, k, v, "NHD", smooth)


def test_prologue_d64_image_size_and_hnd(sage_lib):
    q, k, v = make_qkv(WORKLOADS["B1_H28_S4096_D64"], "cuda")
    _prologue(q, k, v, "NHD", True)
    q, k, v = make_qkv(custom(2, 4, 700, seed_index=1150, k_offset_std=3.0, D=64), "cuda", "HND")
    _prologue(q, k, v, "HND", True)
    q, k, v = make_qkv(custom(2, 5, 1500, seed_index=1151, k_offset_std=3.0, D=64), "cuda", "HND")
    _prologue(q, k, v, "HND", True)


@pytest.mark.parametrize("s_len", [100, 1500])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_prologue_d64_single_head(sage_lib, s_len, layout):
    # one head: the only pair's second head lies past the tensor's head extent
    q, k, v = make_qkv(custom(2, 1, s_len, seed_index=1170 + s_len, k_offset_std=2.0, D=64), "cuda", layout)
    _prologue(q, k, v, layout, True)


@pytest.mark.parametrize("s_len", [300, 1300])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_prologue_d64_head_view_past_the_last_pair(sage_lib, s_len, layout):
    """Heads 0..2 of a 5-head tensor (a view: the head stride and the batch
    stride are the full tensor's). The last pair's second head lies outside
    the view; its memory holds head 3 of the full tensor (large values here),
    which must not leak into any output."""
    w = custom(2, 5, s_len, seed_index=1160 + s_len, k_offset_std=2.0, D=64)
    q, k, v = make_qkv(w, "cuda", layout)
    ax = 2 if layout == "NHD" else 1
    for t in (q, k, v):
        t.narrow(ax, 3, 1).mul_(64.0)  # head 3: never read
    view = [t.narrow(ax, 0, 3) for t in (q, k, v)]
    _prologue(*view, layout, True)

@pytest.mark.parametrize("S,H", [(300, 2), (1300, 3)])
def test_prologue_d64_edge_values(sage_lib, S, H):
    rng = np.random.default_rng(64 + S)
    q = rng.standard_normal((1, S, H, 64)).astype(np.float32)
    k = rng.standard_normal((1, S, H, 64)).astype(np.float32) + 3.0
    v = rng.standard_normal((1, S, H, 64)).astype(np.float32)
    q[0, 32:64, 0] = 0.0
    q[0, 64:96, 0] = -0.0
    q[0, 96:128, 0] = 1e-39                      # subnormal block: the scale is subnormal
    q[0, 128:160, 0] = np.round(rng.uniform(-127, 127, (32, 64)) * 2) / 2   # x / s ties
    q[0, 128, 0, 0] = 127.0
    k[0, 0, 1, 7], k[0, 1, 1, 7], k[0, 2, 1, 7] = 2.0 ** 60, 1.0, -(2.0 ** 60)  # a rounding fp64 chunk sum
    v[0, :, 1, 3] = 0.0
    v[0, :, 1, 4] = -0.0
    v[0, :, 0, 6] = 1e-39
    v[0, 10, 0, 8] = 1e35
    dev = torch.device("cuda")
    qt, kt, vt = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (q, k, v))
    for smooth in (True, False):
        _prologue(qt, kt, vt, "NHD", smooth)


@pytest.mark.parametrize("S", [1000, 2100])
def test_prologue_d64_key_sum_exponent_spread(sage_lib, S):
    # Chunks whose key magnitudes in a channel span 20 to 50 binades: the
    # float-pair chunk sums are taken where they are exact and the fp64 left-to-
    # right sums elsewhere, per channel; ties of x/s and subnormal values mixed in.
    rng = np.random.default_rng(640 + S)
    H = 2
    q = rng.standard_normal((1, S, H, 64)).astype(np.float32)
    k = rng.standard_normal((1, S, H, 64)).astype(np.float32)
    v = rng.standard_normal((1, S, H, 64)).astype(np.float32)
    for c in range(64):
        spread = 20 + (c % 31)
        for chunk in range(0, S, 32):
            n = min(32, S - chunk)
            sign = rng.choice([-1.0, 1.0], n)
            vals = sign * np.ldexp(rng.uniform(1, 2, n), -spread)
            big = rng.integers(0, n)
            vals[big] = sign[big] * rng.uniform(1, 2) * 2.0 ** rng.integers(-2, 3)
            k[0, chunk:chunk + n, c % H, c] = vals
    v[0, 0:64, 1, 5] = np.round(rng.uniform(-448, 448, 64))   # many e4m3 ties once scaled
    v[0, 3, 1, 5] = 448.0
    # a channel on e4m3 rounding boundaries with a power-of-two scale (2^-3)
    e, m = rng.integers(-6, 8, S), rng.integers(8, 16, S)
    v[0, :, 0, 11] = rng.choice([-1.0, 1.0], S) * (2 * m + 1) * np.ldexp(1.0, e - 4) / 8
    v[0, 7, 0, 11] = 56.0
    dev = torch.device("cuda")
    qt, kt, vt = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (q, k, v))
    for smooth in (True, False):
        _prologue(qt, kt, vt, "NHD", smooth)


@pytest.mark.parametrize("s_len", [1, 127, 129, 300, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_d64_matches_oracle(sage_lib, s_len, causal):
    w = custom(1, 3, s_len, seed_index=1200 + s_len, k_offset_std=2.0, D=64)
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", True)
    out, lse = attention(qz, SM64, is_causal=causal, return_lse=True)
    torch.cuda.synchronize()
    assert device_error() == 0 and out.shape == q.shape
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    ref = quantize_tensors(qn, kn, vn, "NHD", True)
    heads = [(0, 0), (0, 1), (0, 2)]
    if not causal:
        check_attention(to_np(out), qn, kn, vn, "NHD", ref, SM64, heads)
    lse_np = lse.cpu().numpy()
    for b, h in heads:
        emu, emu_lse = attention_from_codes(ref, s_len, SM64, b, h, causal=causal, return_lse=True)
        d = np.abs(to_np(out)[b, :, h, :].astype(np.float64) - emu)
        assert d.max() <= 2e-2 and d.mean() <= 2e-3
        assert np.abs(lse_np[b, h].astype(np.float64) - emu_lse).max() <= 2e-4


def test_sageattn_ex_d64_and_page_entry_rejects(sage_lib):
    w = custom(2, 4, 1000, seed_index=1250, k_offset_std=3.0, D=64)
    q, k, v = make_qkv(w, "cuda")
    out, lse = sageattn_ex(q, k, v, is_causal=True, return_lse=True)   # sm_scale None -> 1/8
    torch.cuda.synchronize()
    assert device_error() == 0
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    ref = quantize_tensors(qn, kn, vn, "NHD", True)
    for b, h in [(0, 0), (1, 3)]:
        emu, emu_lse = attention_from_codes(ref, 1000, SM64, b, h, causal=True, return_lse=True, q=qn)
        d = np.abs(to_np(out)[b, :, h, :].astype(np.float64) - emu)
        assert d.max() <= 2e-2 and d.mean() <= 2e-3
        assert np.abs(lse[b, h].cpu().numpy().astype(np.float64) - emu_lse).max() <= 2e-4
    with pytest.raises(SageError):
        sageattn(q, k, v)   # the pages' entry: head dimension 128 only


@pytest.mark.parametrize("s_len", [700, 2100])
def test_sageattn_ex_d64_hnd_repeated(sage_lib, s_len):
    """HND at D = 64 through sageattn_ex, unmasked, called twice with one
    signature (the second call runs from the binding's kept arguments): both
    calls equal, and the output within the tolerances of the oracle's
    emulation on sampled heads, for both prologue kernels."""
    w = custom(2, 5, s_len, seed_index=1270 + s_len, k_offset_std=2.0, D=64)
    q, k, v = make_qkv(w, "cuda", "HND")
    first = sageattn_ex(q, k, v, tensor_layout="HND", sm_scale=SM64)
    again = sageattn_ex(q, k, v, tensor_layout="HND", sm_scale=SM64)
    torch.cuda.synchronize()
    assert device_error() == 0
    assert torch.equal(first, again)
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    ref = quantize_tensors(qn, kn, vn, "HND", True)
    check_attention(to_np(first), qn, kn, vn, "HND", ref, SM64, [(0, 0), (1, 4)])


def test_noalloc_d64_matches_quantize(sage_lib):
    lib = _lib.load()
    w = custom(1, 5, 777, seed_index=1260, k_offset_std=1.0, D=64)
    q, k, v = make_qkv(w, "cuda")
    got = alloc_bundle(1, 777, 5, q.device, 64)
    rc = lib.sage_quantize_noalloc(ctypes.byref(_bf16_tensor(q, "NHD")), ctypes.byref(_bf16_tensor(k, "NHD")),
                                   ctypes.byref(_bf16_tensor(v, "NHD")), 1, 777, 5, 64, 1,
                                   ctypes.byref(got.c_struct()), _stream(q.device))
    assert rc == 0
    ref = quantize(q, k, v, "NHD", True)
    torch.cuda.synchronize()
    assert_bundles_equal(bundle_np(got), bundle_np(ref))


def test_d64_video_size_sampled_rows(sage_lib):
    w = WORKLOADS["B1_H28_S16384_D64"]
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", True)
    out = attention(qz, SM64)
    torch.cuda.synchronize()
    assert device_error() == 0
    heads = [(0, 0), (0, 27)]
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    ref = quantize_tensors(qn, kn, vn, "NHD", True, heads=heads)
    assert_bundles_equal(bundle_np(qz), ref, heads=heads)
    rows = np.sort(np.random.default_rng(5).choice(16384, 100, replace=False))
    check_attention(to_np(out), qn, kn, vn, "NHD", ref, SM64, heads, rows=rows)
