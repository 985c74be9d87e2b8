"""Failure detection on the GPU without a fault: a bounded wait that runs out.

sage_selftest_wait_timeout launches one warp that waits, with the same
bounded wait the library's kernels use, on a barrier nothing completes. After
the wait's 2 s limit the kernel sets the device error word and returns; the
host reads SAGE_ERR_DEVICE_TIMEOUT, and the context still runs an ordinary
call correctly. Nothing traps or hangs.
"""

import math
import time

import numpy as np
import pytest
import torch

from gpu_util import check_attention, to_np
from oracle.tensors import quantize_tensors
from quantized_attention_fp64_gb300 import _lib, device_error, sageattn
from quantized_attention_fp64_gb300.api import _stream_handle
from quantized_attention_fp64_gb300.workloads import custom, make_qkv

pytestmark = pytest.mark.gpu
SAGE_ERR_DEVICE_TIMEOUT = -12


def test_bounded_wait_runs_out_and_the_context_stays_usable(sage_lib):
    lib = _lib.load()
    torch.cuda.synchronize()
    assert device_error() == 0  # reads and clears the word
    t0 = time.monotonic()
    assert lib.sage_selftest_wait_timeout(_stream_handle(torch.cuda.current_device())) == 0
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert device_error() == SAGE_ERR_DEVICE_TIMEOUT
    assert device_error() == 0  # cleared by the read
    assert 1.5 <= waited <= 30.0, waited
    # an ordinary call afterwards, checked against the oracle
    w = custom(1, 2, 300, seed_index=901, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda")
    sm = 1.0 / math.sqrt(128.0)
    out = sageattn(q, k, v, sm_scale=sm)
    torch.cuda.synchronize()
    assert device_error() == 0
    qn, kn, vn = to_np(q), to_np(k), to_np(v)
    ref = quantize_tensors(qn, kn, vn, "NHD", True)
    check_attention(to_np(out), qn, kn, vn, "NHD", ref, sm, [(0, 0), (0, 1)])
    assert np.isfinite(to_np(out)).all()
