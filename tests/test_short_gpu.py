"""Short sequences (S <= 1024): the prologue runs as one cluster of
ceil(S / 128) CTAs per head, exchanging the group key sums and V maxima
through distributed shared memory; longer sequences run the persistent
kernel. Both must give the oracle's bundle bit for bit, on either side of the
threshold, for every cluster size, and with many clusters in flight. The
attention kernel is launched as a programmatic dependent of the kernel before
it: it must still see that kernel's writes, whoever launched it.
"""

import math

import numpy as np
import pytest
import torch

from gpu_util import assert_bundles_equal, bundle_np, check_attention, to_np
from oracle.tensors import quantize_tensors
from quantized_attention_fp64_gb300 import attention, device_error, quantize, sageattn
from quantized_attention_fp64_gb300.workloads import custom, make_qkv

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(128.0)


def _bundle_matches(q, k, v, layout, smooth, heads=None):
    qz = quantize(q, k, v, layout, smooth)
    torch.cuda.synchronize()
    assert device_error() == 0
    ref = quantize_tensors(to_np(q), to_np(k), to_np(v), layout, smooth, heads=heads)
    assert_bundles_equal(bundle_np(qz), ref, heads=heads)
    return qz


@pytest.mark.parametrize("s_len", [1, 127, 128, 129, 384, 640, 768, 897, 1023, 1024, 1025, 1152])
@pytest.mark.parametrize("smooth", [True, False])
def test_prologue_every_cluster_size(sage_lib, s_len, smooth):
    # 1 .. 8 groups per head (short kernel), then 9 and 9 (persistent kernel)
    w = custom(2, 3, s_len, seed_index=3000 + s_len, k_offset_std=2.5)
    q, k, v = make_qkv(w, "cuda")
    _bundle_matches(q, k, v, "NHD", smooth)


def test_prologue_short_hnd_and_strided(sage_lib):
    w = custom(2, 5, 700, seed_index=3100, k_offset_std=1.5)
    q, k, v = make_qkv(w, "cuda", "HND")
    _bundle_matches(q, k, v, "HND", True)
    # a view with a padded head stride (NHD, heads 0..3 of 6)
    w = custom(1, 6, 333, seed_index=3101, k_offset_std=1.5)
    q, k, v = make_qkv(w, "cuda")
    _bundle_matches(q[:, :, :4], k[:, :, :4], v[:, :, :4], "NHD", True)


def test_prologue_short_many_clusters(sage_lib):
    # 4 x 80 heads x 7 groups: far more clusters than fit on the GPU at once
    w = custom(4, 80, 833, seed_index=3200, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda")
    _bundle_matches(q, k, v, "NHD", True, heads=[(0, 0), (1, 41), (3, 79)])


@pytest.mark.parametrize("s_len", [300, 1300])
def test_prologue_edge_values_both_kernels(sage_lib, s_len):
    """Zero, negative-zero and subnormal blocks, x/s ties, a key chunk whose
    fp64 sum rounds, tiny keys beside a huge one and a huge V value, through
    the short kernel (300 tokens) and the persistent one (1300)."""
    rng = np.random.default_rng(17 + s_len)
    H = 2
    q = rng.standard_normal((1, s_len, H, 128)).astype(np.float32)
    k = rng.standard_normal((1, s_len, H, 128)).astype(np.float32) + 3.0
    v = rng.standard_normal((1, s_len, H, 128)).astype(np.float32)
    q[0, 32:64, 0] = 0.0
    q[0, 64:96, 0] = -0.0
    q[0, 96:128, 0] = 1e-39
    q[0, 128:160, 0] = np.round(rng.uniform(-127, 127, (32, 128)) * 2) / 2
    k[0, 0, 1, 7], k[0, 1, 1, 7], k[0, 2, 1, 7] = 2.0 ** 60, 1.0, -(2.0 ** 60)
    k[0, 200:232, 1, 9] = 1e-38
    k[0, 200, 1, 9] = 1e30
    v[0, :, 1, 3] = 0.0
    v[0, :, 1, 4] = -0.0
    v[0, :, 0, 6] = 1e-39
    v[0, s_len - 1, 0, 8] = 1e35
    dev = torch.device("cuda")
    qt, kt, vt = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (q, k, v))
    for smooth in (True, False):
        _bundle_matches(qt, kt, vt, "NHD", smooth)


@pytest.mark.parametrize("s_len", [1000, 2100])
def test_key_sum_exponent_spread_both_kernels(sage_lib, s_len):
    """Key chunks spanning 20 to 50 binades (float-pair sums and the fp64
    fallback both run), in the short kernel and in the persistent one."""
    rng = np.random.default_rng(23 + s_len)
    H = 2
    q = rng.standard_normal((1, s_len, H, 128)).astype(np.float32)
    k = rng.standard_normal((1, s_len, H, 128)).astype(np.float32)
    v = rng.standard_normal((1, s_len, H, 128)).astype(np.float32)
    for c in range(128):
        spread = 20 + (c % 31)
        for chunk in range(0, s_len, 32):
            n = min(32, s_len - chunk)
            sign = rng.choice([-1.0, 1.0], n)
            vals = sign * np.ldexp(rng.uniform(1, 2, n), -spread)
            big = rng.integers(0, n)
            vals[big] = sign[big] * rng.uniform(1, 2) * 2.0 ** rng.integers(-2, 3)
            k[0, chunk:chunk + n, c % H, c] = vals
    dev = torch.device("cuda")
    qt, kt, vt = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (q, k, v))
    _bundle_matches(qt, kt, vt, "NHD", True)


def _e4m3_midpoints(rng, n, scale):
    """n values v with v / scale exactly halfway between two e4m3 values
    (below 448, so that the channel maximum 448 * scale sets the scale)."""
    e = rng.integers(-6, 8, n)
    m = rng.integers(8, 16, n)
    sign = rng.choice([-1.0, 1.0], n)
    return sign * (2 * m + 1) * np.ldexp(1.0, e - 4) * scale


@pytest.mark.parametrize("s_len", [300, 1300])
def test_v_code_ties_both_kernels(sage_lib, s_len):
    """V channels whose scale is a power of two (max |v| = 448 * 2^k) filled
    with values on e4m3 rounding boundaries: the fast brackets straddle every
    one of them, and the exact quotient must round half to even."""
    rng = np.random.default_rng(31 + s_len)
    H = 2
    q = rng.standard_normal((1, s_len, H, 128)).astype(np.float32)
    k = rng.standard_normal((1, s_len, H, 128)).astype(np.float32)
    v = rng.standard_normal((1, s_len, H, 128)).astype(np.float32)
    for c, scale in ((3, 1.0), (40, 0.125), (77, 2.0 ** -20), (127, 64.0)):
        col = _e4m3_midpoints(rng, s_len, scale)
        col[s_len // 2] = 448.0 * scale
        v[0, :, c % H, c] = col
    dev = torch.device("cuda")
    qt, kt, vt = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (q, k, v))
    _bundle_matches(qt, kt, vt, "NHD", True)


@pytest.mark.parametrize("s_len", [96, 256, 1000])
def test_sageattn_short_matches_oracle(sage_lib, s_len):
    w = custom(2, 4, s_len, seed_index=3300 + s_len, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda")
    out = sageattn(q, k, v, sm_scale=SM)
    torch.cuda.synchronize()
    assert device_error() == 0
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    ref = quantize_tensors(qn, kn, vn, "NHD", True)
    check_attention(to_np(out), qn, kn, vn, "NHD", ref, SM, [(0, 0), (1, 3)])


def test_attention_waits_for_the_kernel_before_it(sage_lib):
    # The attention kernel may start before the previous kernel of the stream
    # ends; it must not read the bundle before that kernel's writes land. A
    # torch kernel rewrites the key copies and V codes right before the call.
    w = custom(1, 8, 1000, seed_index=3400, k_offset_std=1.0)
    q, k, v = make_qkv(w, "cuda")
    qz = quantize(q, k, v, "NHD", True)
    torch.cuda.synchronize()
    k16_saved, vt_saved = qz.k16.clone(), qz.vt_codes.clone()
    for rep in range(3):
        qz.k16.copy_(torch.flip(k16_saved, dims=[2]))
        qz.vt_codes.copy_(torch.flip(vt_saved, dims=[3]))
        got = attention(qz, SM)                      # no synchronize in between
        torch.cuda.synchronize()
        want = attention(qz, SM)                     # inputs settled
        torch.cuda.synchronize()
        assert torch.equal(got, want)
        qz.k16.copy_(k16_saved)
        qz.vt_codes.copy_(vt_saved)
        got = attention(qz, SM)
        torch.cuda.synchronize()
        want = attention(qz, SM)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    assert device_error() == 0


def test_back_to_back_calls_on_one_stream(sage_lib):
    # many short calls queued without synchronizing: each result must equal
    # the one computed alone
    outs, inputs = [], []
    for i in range(6):
        w = custom(1, 4, 200 + 150 * i, seed_index=3500 + i, k_offset_std=1.0)
        inputs.append(make_qkv(w, "cuda"))
    torch.cuda.synchronize()
    for q, k, v in inputs:
        outs.append(sageattn(q, k, v, sm_scale=SM))
    torch.cuda.synchronize()
    for (q, k, v), o in zip(inputs, outs):
        alone = sageattn(q, k, v, sm_scale=SM)
        torch.cuda.synchronize()
        assert torch.equal(o, alone)
    assert device_error() == 0


def test_sageattn_short_reuses_one_workspace(sage_lib):
    # calls that reuse one workspace (new inputs each time, and a torch
    # kernel rewriting the inputs right before a call) must each see only
    # their own prologue's output
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    shapes = [(1, 4, 256), (2, 3, 700), (1, 4, 256), (1, 8, 1024)]
    inputs = [make_qkv(custom(b, h, s, seed_index=3600 + i, k_offset_std=1.0), "cuda")
              for i, (b, h, s) in enumerate(shapes)]
    alone = []
    for q, k, v in inputs:
        alone.append(sageattn(q, k, v, sm_scale=SM))
        torch.cuda.synchronize()
    outs = [sageattn(q, k, v, sm_scale=SM, workspace=ws) for q, k, v in inputs]
    q, k, v = inputs[0]
    q2 = q.clone()
    q2.mul_(-1.0)                                     # torch kernel right before the call
    neg = sageattn(q2, k, v, sm_scale=SM, workspace=ws)
    torch.cuda.synchronize()
    for o, a in zip(outs, alone):
        assert torch.equal(o, a)
    assert torch.equal(neg, sageattn(-q, k, v, sm_scale=SM))
    assert device_error() == 0


def test_repeated_signature_takes_prepared_arguments(sage_lib):
    """A call whose shapes, strides, dtypes, devices, layout and flags were seen
    before runs from the kept arguments: it must give the first call's result
    bit for bit, honour a new sm_scale and new inputs, keep layouts and flags
    apart, and still reject tensors that differ from the kept signature."""
    from quantized_attention_fp64_gb300 import SageError, api, sageattn_ex

    calls = api._forget_calls()
    w = custom(2, 4, 384, seed_index=3600, k_offset_std=1.5)
    q, k, v = make_qkv(w, "cuda")
    first = sageattn(q, k, v, sm_scale=SM)
    assert len(calls) == 1
    again = sageattn(q, k, v, sm_scale=SM)
    other_scale = sageattn(q, k, v, sm_scale=0.5 * SM)
    q2, k2, v2 = make_qkv(custom(2, 4, 384, seed_index=3601, k_offset_std=0.5), "cuda")
    fresh = sageattn(q2, k2, v2, sm_scale=SM)
    torch.cuda.synchronize()
    assert torch.equal(first, again)
    api._forget_calls()
    assert torch.equal(other_scale, sageattn(q, k, v, sm_scale=0.5 * SM))
    api._forget_calls()
    assert torch.equal(fresh, sageattn(q2, k2, v2, sm_scale=SM))
    # causal and the LSE through the ex entry point, twice each
    c1 = sageattn_ex(q, k, v, is_causal=True, sm_scale=SM)
    c2 = sageattn_ex(q, k, v, is_causal=True, sm_scale=SM)
    o1, l1 = sageattn_ex(q, k, v, sm_scale=SM, return_lse=True)
    o2, l2 = sageattn_ex(q, k, v, sm_scale=SM, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2) and torch.equal(o1, o2) and torch.equal(l1, l2)
    assert not torch.equal(c1, first)
    # the same sizes in HND (other strides) and a padded-stride view
    qh, kh, vh = (t.transpose(1, 2).contiguous() for t in (q, k, v))
    h1 = sageattn(qh, kh, vh, tensor_layout="HND", sm_scale=SM)
    h2 = sageattn(qh, kh, vh, tensor_layout="HND", sm_scale=SM)
    torch.cuda.synchronize()
    assert torch.equal(h1, h2) and torch.equal(h1.transpose(1, 2), first)
    # tensors that differ from a kept signature take the full checks
    with pytest.raises((SageError, ValueError)):
        sageattn(q, k.cpu(), v, sm_scale=SM)
    with pytest.raises(SageError):
        sageattn(q, k.to(torch.float16), v, sm_scale=SM)
    with pytest.raises(SageError):
        sageattn(q, k[:, :200], v[:, :200], sm_scale=SM)
    assert device_error() == 0


def test_two_threads_on_one_stream(sage_lib):
    """Two threads calling sageattn at once on the same stream (the library
    call releases the GIL, so their launches interleave): every result must
    equal the one computed alone."""
    import threading

    inputs = [make_qkv(custom(1, 4, 256 + 128 * (i % 3), seed_index=3700 + i, k_offset_std=1.0), "cuda")
              for i in range(6)]
    torch.cuda.synchronize()
    alone = []
    for q, k, v in inputs:
        alone.append(sageattn(q, k, v, sm_scale=SM))
        torch.cuda.synchronize()
    results = {}
    errors = []

    def worker(t):
        try:
            outs = []
            for rep in range(40):
                i = (t + 2 * rep) % len(inputs)
                outs.append((i, sageattn(*inputs[i], sm_scale=SM)))
            results[t] = outs
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    torch.cuda.synchronize()
    assert not errors and len(results) == 2
    for outs in results.values():
        for i, o in outs:
            assert torch.equal(o, alone[i])
    assert device_error() == 0
