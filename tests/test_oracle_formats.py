"""Pins for the oracle's number formats: bf16 rounding and the e4m3fn codec.

Each check ties the oracle to something outside itself: hand-derived values
from the format definitions (tests/golden/), PyTorch's own conversions, CUDA's
host-side FP8 conversion, and brute-force search over the e4m3 value set.
"""

import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

from oracle import bf16_round, e4m3_decode, e4m3_encode
from pin_util import e4m3_round_bruteforce

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden_e4m3():
    rows = []
    with open(os.path.join(HERE, "golden", "e4m3fn_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            rows.append((int(code, 16), float(val)))
    return rows


def _structured_f32(lo_exp=-14, hi_exp=9, seed=0):
    """Float32 values around every e4m3 value and every midpoint between two
    neighbouring e4m3 values (+-0..3 float32 steps), over both signs, plus
    random values spread over [2^lo_exp, 2^hi_exp)."""
    vals = e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)).astype(np.float32)
    mids = ((vals[:-1].astype(np.float64) + vals[1:].astype(np.float64)) / 2).astype(np.float32)
    base = np.concatenate([vals, mids])
    out = [base]
    for k in range(1, 4):
        up, dn = base.copy(), base.copy()
        for _ in range(k):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(-np.inf))
        out += [up, dn]
    rng = np.random.default_rng(seed)
    out.append((2.0 ** rng.uniform(lo_exp, hi_exp, 20000)).astype(np.float32))
    pos = np.concatenate(out)
    pos = pos[pos >= 0]
    return np.concatenate([pos, -pos]).astype(np.float32)


def test_bf16_round_hand_cases():
    # bf16 keeps 7 mantissa bits: 1 + 2^-8 is a tie between 1 and 1 + 2^-7 and
    # goes to the even mantissa (1.0); 1 + 3*2^-8 ties between 1 + 2^-7 (odd)
    # and 1 + 2^-6 (even).
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1 + 2 ** -8 + 2 ** -20], np.float32)
    assert bf16_round(x).tolist() == [1.0, 1.015625, -1.0, 1.0078125]


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # exact ties: upper 16 bits random, lower 16 bits = 0x8000
    ties = ((rng.integers(0, 2 ** 16, 5000, dtype=np.uint64) << 16) | 0x8000).astype(np.uint32).view(np.float32)
    ties = ties[np.isfinite(ties)]
    x = np.concatenate([x, ties, np.array([0.0, -0.0, 1e-40, -1e-40, 3.4e38], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = bf16_round(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_e4m3_decode_golden():
    for code, val in _golden_e4m3():
        got = float(e4m3_decode(np.array([code], np.uint8))[0])
        if np.isnan(val):
            assert np.isnan(got), hex(code)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), hex(code)


def test_e4m3_encode_golden_roundtrip():
    for code, val in _golden_e4m3():
        if np.isnan(val):
            continue
        assert int(e4m3_encode(np.array([val], np.float32))[0]) == code, hex(code)


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_encode_hand_cases():
    # satfinite: everything from 448 up saturates (464 is the tie between 448,
    # mantissa 110, and the absent 480, mantissa 111: even wins); ties in the
    # subnormal range go to the even code.
    cases = [(448.0, 0x7E), (460.0, 0x7E), (464.0, 0x7E), (470.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE),
             (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (5 * 2.0 ** -10, 0x02), (2.0 ** -11, 0x00),
             (-(2.0 ** -11), 0x80), (0.0, 0x00), (-0.0, 0x80), (1.0625, 0x38), (1.1875, 0x3A),
             (float("inf"), 0x7E), (float("-inf"), 0xFE)]
    xs = np.array([x for x, _ in cases], np.float32)
    got = e4m3_encode(xs)
    for (x, c), g in zip(cases, got):
        assert int(g) == c, (x, hex(c), hex(int(g)))


def test_e4m3_encode_matches_torch_in_range():
    x = _structured_f32()
    x = x[np.abs(x) <= 464.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = e4m3_encode(x)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(x[i]), hex(ref[i]), hex(got[i])) for i in bad[:10]]


def test_e4m3_encode_bruteforce_sample():
    x = _structured_f32(seed=2)
    rng = np.random.default_rng(3)
    sample = np.concatenate([x[rng.integers(0, x.size, 3000)],
                             np.array([500.0, -1000.0, 449.0, 463.99, 464.01], np.float32)])
    got = e4m3_encode(sample)
    for xv, g in zip(sample, got):
        assert int(g) == e4m3_round_bruteforce(float(xv)), float(xv)


def test_e4m3_encode_matches_cuda_host_conversion():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    x = np.concatenate([_structured_f32(seed=4),
                        np.array([448.0, 464.0, 465.0, 1e6, -1e6, 3e38, -0.0], np.float32)])
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "cvt")
        subprocess.run([nvcc, "-O2", "-o", exe, os.path.join(HERE, "helpers", "fp8_host_cvt.cu")],
                       check=True, capture_output=True)
        fin, fout = os.path.join(d, "in.bin"), os.path.join(d, "out.bin")
        x.tofile(fin)
        subprocess.run([exe, fin, fout], check=True)
        ref = np.fromfile(fout, dtype=np.uint8)
    got = e4m3_encode(x)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(x[i]), hex(ref[i]), hex(got[i])) for i in bad[:10]]
