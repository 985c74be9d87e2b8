"""sage_sageattn_host: host-resident inputs and output, the head groups'
copies overlapping the kernels of the other groups. Every head is computed
by the same kernels as on device tensors, so the output must equal
sage_sageattn_ex's on the same inputs bit for bit, whatever the grouping,
layout, head dimension or memory kind, and in back-to-back calls."""

import math

import pytest
import torch

from quantized_attention_fp64_gb300 import device_error, sageattn_ex, sageattn_host
from quantized_attention_fp64_gb300.workloads import WORKLOADS, custom, make_qkv

pytestmark = pytest.mark.gpu


def _host(t, pinned=True):
    h = t.cpu()
    return h.pin_memory() if pinned else h


def _expect(q, k, v, layout, causal, sm, smooth=True):
    out = sageattn_ex(q, k, v, tensor_layout=layout, is_causal=causal, sm_scale=sm, smooth_k=smooth)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("n_groups", [0, 1, 2, 5])
def test_host_matches_device_nhd(sage_lib, n_groups):
    w = custom(2, 5, 700, seed_index=4000, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda")
    sm = 1.0 / math.sqrt(128.0)
    want = _expect(q, k, v, "NHD", False, sm)
    got = sageattn_host(_host(q), _host(k), _host(v), sm_scale=sm, n_groups=n_groups)
    torch.cuda.synchronize()
    assert device_error() == 0
    assert torch.equal(got, want)


@pytest.mark.parametrize("causal", [False, True])
def test_host_matches_device_hnd_and_d64(sage_lib, causal):
    for D, S in ((128, 1500), (64, 900)):
        w = custom(2, 3, S, seed_index=4100 + D, k_offset_std=1.5, D=D)
        q, k, v = make_qkv(w, "cuda", "HND")
        want = _expect(q, k, v, "HND", causal, None)
        got = sageattn_host(_host(q), _host(k), _host(v), tensor_layout="HND", is_causal=causal, n_groups=2)
        torch.cuda.synchronize()
        assert device_error() == 0
        assert torch.equal(got, want), (D, S)


def test_host_pageable_memory_and_smooth_off(sage_lib):
    w = custom(1, 4, 333, seed_index=4200, k_offset_std=3.0)
    q, k, v = make_qkv(w, "cuda")
    want = _expect(q, k, v, "NHD", False, 0.05, smooth=False)
    got = sageattn_host(_host(q, False), _host(k, False), _host(v, False), sm_scale=0.05, smooth_k=False,
                        n_groups=3)
    torch.cuda.synchronize()
    assert torch.equal(got, want)


def test_host_back_to_back_reusing_buffers(sage_lib):
    # several calls queued on one stream with one workspace and one output
    # buffer per call: each result equals its device counterpart
    sm = 1.0 / math.sqrt(128.0)
    cases = []
    for i in range(3):
        w = custom(1, 6, 500 + 400 * i, seed_index=4300 + i, k_offset_std=1.0)
        q, k, v = make_qkv(w, "cuda")
        cases.append(((q, k, v), tuple(_host(t) for t in (q, k, v))))
    ws = torch.empty(1 << 28, dtype=torch.uint8, device="cuda")
    outs = [sageattn_host(*h, sm_scale=sm, workspace=ws, n_groups=2) for _, h in cases]
    torch.cuda.synchronize()
    for (dev, _), got in zip(cases, outs):
        assert torch.equal(got, _expect(*dev, "NHD", False, sm))
    assert device_error() == 0


def test_host_video_size(sage_lib):
    # the benchmark workload, grouped as the library chooses
    w = WORKLOADS["B1_H28_S16384"]
    q, k, v = make_qkv(w, "cuda")
    sm = 1.0 / math.sqrt(128.0)
    want = _expect(q, k, v, "NHD", False, sm)
    got = sageattn_host(_host(q), _host(k), _host(v), sm_scale=sm)
    torch.cuda.synchronize()
    assert device_error() == 0
    assert torch.equal(got, want)
