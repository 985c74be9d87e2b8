"""sage_quantize_noalloc: the quantization prologue for callers that cannot
allocate device memory (code held to a memory budget fixed up front, plug-ins
handed only the tensors they read and write, hosts whose allocator must not be
entered from the calling thread). It keeps its scratch in a device array built
into the library instead of a caller-provided buffer.

Checked through the C ABI against sage_quantize (which takes a caller-owned
scratch buffer): the codes, scales and key means must be identical, bit for
bit, as every prologue result is. Several problems run back to back, so each
call also shows that what the previous one left in the shared array does not
leak into its result: at D = 128 sequences longer than 1024 tokens take the
persistent prologue, which keeps its work counter, per-head flags and partial
sums in that array, and shorter ones take the cluster kernel, which uses none
of it (one runs between two persistent calls). This file sorts last so that a
run stopping at the first failure has already run every other test."""

import ctypes

import pytest
import torch

from gpu_util import assert_bundles_equal, bundle_np
from quantized_attention_fp64_gb300 import _lib
from quantized_attention_fp64_gb300.api import _bf16_tensor, _stream, alloc_bundle, quantize
from quantized_attention_fp64_gb300.workloads import custom, make_qkv

pytestmark = pytest.mark.gpu

SAGE_ERR_WORKSPACE = -9
SAGE_ERR_TOO_LARGE = -14


def _noalloc(lib, q, k, v, smooth_k):
    B, S, H, D = q.shape
    qz = alloc_bundle(B, S, H, q.device, D)
    bundle = qz.c_struct()
    rc = lib.sage_quantize_noalloc(ctypes.byref(_bf16_tensor(q, "NHD")), ctypes.byref(_bf16_tensor(k, "NHD")),
                                   ctypes.byref(_bf16_tensor(v, "NHD")), B, S, H, D, int(smooth_k),
                                   ctypes.byref(bundle), _stream(q.device))
    assert rc == 0, lib.sage_strerror(rc)
    return qz


def test_noalloc_matches_quantize_twice(sage_lib):
    lib = _lib.load()
    problems = [(custom(2, 8, 1024, seed_index=901, k_offset_std=3.0), True),
                (custom(1, 5, 777, seed_index=902, k_offset_std=1.0), False)]
    for w, smooth in problems:
        q, k, v = make_qkv(w, "cuda")
        got = _noalloc(lib, q, k, v, smooth)
        ref = quantize(q, k, v, "NHD", smooth)
        torch.cuda.synchronize()
        assert_bundles_equal(bundle_np(got), bundle_np(ref))


def test_noalloc_persistent_path_back_to_back(sage_lib):
    """Two persistent-kernel problems (S > 1024) through the built-in scratch,
    with a cluster-kernel call between them: the second persistent call must
    not see the first one's counters, flags or partial sums."""
    lib = _lib.load()
    problems = [(custom(1, 4, 2200, seed_index=903, k_offset_std=2.0), True),
                (custom(1, 3, 300, seed_index=904, k_offset_std=2.0), True),
                (custom(2, 3, 1500, seed_index=905, k_offset_std=0.0), False),
                (custom(1, 4, 2200, seed_index=906, k_offset_std=2.0), True),
                # head dimension 64: head pairs, with an odd head count (the
                # scratch also holds each pair's key mean and V scales)
                (custom(2, 5, 1700, seed_index=907, k_offset_std=2.0, D=64), True),
                (custom(1, 4, 2200, seed_index=908, k_offset_std=1.0), True)]
    for w, smooth in problems:
        q, k, v = make_qkv(w, "cuda")
        got = _noalloc(lib, q, k, v, smooth)
        ref = quantize(q, k, v, "NHD", smooth)
        torch.cuda.synchronize()
        assert_bundles_equal(bundle_np(got), bundle_np(ref))


def test_noalloc_rejects_problems_beyond_its_buffer(sage_lib):
    lib = _lib.load()
    q = torch.zeros(1, 64, 2, 128, dtype=torch.bfloat16, device="cuda")
    qz = alloc_bundle(1, 64, 2, q.device)
    bundle = qz.c_struct()
    t = _bf16_tensor(q, "NHD")
    # 80 heads x 131072 tokens need about 120 MiB of scratch, over the 32 MiB
    # built in; the call is refused before anything is launched
    rc = lib.sage_quantize_noalloc(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), 1, 131072, 80, 128, 1,
                                   ctypes.byref(bundle), _stream(q.device))
    assert rc == SAGE_ERR_WORKSPACE
    # sizes past the library's general limits are refused like sage_quantize's
    rc = lib.sage_quantize_noalloc(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), 65535, 1 << 20, 65535, 128,
                                   1, ctypes.byref(bundle), _stream(q.device))
    assert rc == SAGE_ERR_TOO_LARGE
