"""GPU prologue against the oracle: INT8 Q/K codes, e4m3 V codes, every scale
and the key mean must match bit for bit."""

import numpy as np
import pytest
import torch

from gpu_util import assert_bundles_equal, bundle_np, to_np
from oracle.tensors import quantize_tensors
from quantized_attention_fp64_gb300 import quantize
from quantized_attention_fp64_gb300.workloads import WORKLOADS, custom, make_qkv

pytestmark = pytest.mark.gpu


def _run(q, k, v, layout, smooth, heads=None):
    qz = quantize(q, k, v, layout, smooth)
    torch.cuda.synchronize()
    ref = quantize_tensors(to_np(q), to_np(k), to_np(v), layout, smooth, heads=heads)
    assert_bundles_equal(bundle_np(qz), ref, heads=heads)


@pytest.mark.parametrize("name,smooth,layout", [
    ("B1_H2_S256", False, "NHD"), ("B1_H2_S256", True, "NHD"),
    ("B2_H8_S1024", True, "NHD"), ("B2_H8_S1024", False, "NHD"), ("B2_H8_S1024", True, "HND"),
    ("B1_H28_S4096", True, "NHD"),
])
def test_prologue_configs(sage_lib, name, smooth, layout):
    q, k, v = make_qkv(WORKLOADS[name], "cuda", layout)
    _run(q, k, v, layout, smooth)


@pytest.mark.parametrize("s_len", [1, 31, 33, 129, 255, 257, 1000, 4097])
def test_prologue_ragged_lengths(sage_lib, s_len):
    w = custom(2, 3, s_len, seed_index=200 + s_len, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda")
    _run(q, k, v, "NHD", True)


def test_prologue_full_video_size(sage_lib):
    q, k, v = make_qkv(WORKLOADS["B1_H28_S16384"], "cuda")
    _run(q, k, v, "NHD", True)


def test_prologue_long_sequence_sampled_heads(sage_lib):
    # Past 100k tokens (the length that used to need 64-bit offsets); the
    # oracle checks three heads in full.
    q, k, v = make_qkv(WORKLOADS["B1_H28_S131072"], "cuda")
    _run(q, k, v, "NHD", True, heads=[(0, 0), (0, 13), (0, 27)])


@pytest.mark.parametrize("S", [300, 1300])
def test_prologue_edge_values(sage_lib, S):
    """Zero blocks and channels, negative zeros, bf16 subnormals, exact .5
    ties of x/s, a key chunk whose fp64 sum rounds (forcing the exact fp64
    path) and huge magnitudes; S = 300 runs the cluster kernel, S = 1300 the
    persistent one (whose head key sums then take the pairwise tree over the
    group sums)."""
    rng = np.random.default_rng(5)
    H = 2
    q = rng.standard_normal((1, S, H, 128)).astype(np.float32)
    k = rng.standard_normal((1, S, H, 128)).astype(np.float32) + 3.0
    v = rng.standard_normal((1, S, H, 128)).astype(np.float32)
    q[0, 32:64, 0] = 0.0                       # zero Q block
    q[0, 64:96, 0] = -0.0                      # negative-zero Q block
    q[0, 96:128, 0] = 1e-39                    # subnormal bf16 block: s is subnormal
    q[0, 96, 0, 5] = 3e-39
    q[0, 128:160, 0] = np.round(rng.uniform(-127, 127, (32, 128)) * 2) / 2   # x/s ties
    q[0, 128, 0, 0] = 127.0
    k[0, 0, 1, 7], k[0, 1, 1, 7], k[0, 2, 1, 7] = 2.0 ** 60, 1.0, -(2.0 ** 60)   # rounding fp64 chunk sum
    k[0, 40:72, 1, 9] = 1e-38                  # tiny values beside large ones
    k[0, 40, 1, 9] = 1e30
    v[0, :, 1, 3] = 0.0                        # zero V channel
    v[0, :, 1, 4] = -0.0                       # negative-zero V channel
    v[0, :, 0, 6] = 1e-39                      # subnormal V channel: s_v subnormal
    v[0, 7, 0, 6] = -2e-39
    v[0, 10, 0, 8] = 1e35                      # one huge value dominates its channel
    dev = torch.device("cuda")
    qt, kt, vt = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (q, k, v))
    for smooth in (True, False):
        _run(qt, kt, vt, "NHD", smooth)


@pytest.mark.parametrize("S", [1000, 2100])
def test_prologue_key_sum_exponent_spread(sage_lib, S):
    """Key chunks whose magnitudes span 20 to 50 binades, so that both the
    float-pair chunk sums and the fp64 fallback run, with cancelling signs and
    ragged chunks; the key mean and every code must still match bit for bit
    (S = 1000: the cluster kernel; S = 2100: the persistent kernel)."""
    rng = np.random.default_rng(11)
    H = 3
    q = rng.standard_normal((1, S, H, 128)).astype(np.float32)
    k = rng.standard_normal((1, S, H, 128)).astype(np.float32)
    v = rng.standard_normal((1, S, H, 128)).astype(np.float32)
    for c in range(128):
        spread = 20 + (c % 31)                     # exponent gap between big and tiny entries
        for chunk in range(0, S, 32):
            rows = slice(chunk, min(chunk + 32, S))
            n = min(32, S - chunk)
            sign = rng.choice([-1.0, 1.0], n)
            big = rng.integers(0, n)
            vals = sign * np.ldexp(rng.uniform(1, 2, n), -spread)
            vals[big] = sign[big] * rng.uniform(1, 2) * 2.0 ** rng.integers(-2, 3)
            k[0, rows, c % H, c] = vals
    dev = torch.device("cuda")
    qt, kt, vt = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (q, k, v))
    _run(qt, kt, vt, "NHD", True)
    _run(qt, kt, vt, "NHD", False)


@pytest.mark.parametrize("S", [256, 2048])
def test_prologue_chunk_bounds_second_half(sage_lib, S):
    """A key chunk whose exponent spread sits only in the second half of its
    32 tokens, in channels past the first 8: tokens 16, 18, 20 of the chunk
    hold 1, 2^-24 and 2^-52 in one channel that is zero elsewhere. The
    float-pair chunk sum loses the 2^-52 (its error term rounds), the
    left-to-right fp64 sum keeps it, and the key mean fl32(T / S) then sits
    just above an fp32 tie instead of on it; each warp's exactness test must
    use the bounds of its own channels from the other half's rows."""
    rng = np.random.default_rng(23)
    H = 2
    q = rng.standard_normal((1, S, H, 128)).astype(np.float32)
    k = rng.standard_normal((1, S, H, 128)).astype(np.float32)
    v = rng.standard_normal((1, S, H, 128)).astype(np.float32)
    for h, c, chunk in ((0, 8, 0), (1, 77, 5)):
        t0 = 32 * chunk + 16
        k[0, :, h, c] = 0.0
        k[0, t0, h, c], k[0, t0 + 2, h, c], k[0, t0 + 4, h, c] = 1.0, 2.0 ** -24, 2.0 ** -52
    dev = torch.device("cuda")
    qt, kt, vt = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (q, k, v))
    _run(qt, kt, vt, "NHD", True)
