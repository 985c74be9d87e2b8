"""The C ABI without a GPU: the library loads, exports every function the
header declares, answers size queries, and rejects invalid calls before it
touches the device (every case here has an argument the host validation
refuses, so nothing is ever launched)."""

import ctypes
import math

import pytest
import torch

from quantized_attention_fp64_gb300 import _build, _lib
from quantized_attention_fp64_gb300.api import SageError, sageattn

OK, CAUSAL, LSE, DTYPE, HEAD_DIM, SHAPE, LAYOUT, ALIGN, NULLPTR, WORKSPACE = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9
ARG, TOO_LARGE = -13, -14


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _lib.header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_strerror_covers_codes(lib):
    for code in range(0, -16, -1):
        msg = lib.sage_strerror(code)
        assert msg and b"unknown" not in msg
    assert b"unknown" in lib.sage_strerror(-99)


def _sizes(lib, fn, *args):
    n = ctypes.c_size_t(0)
    rc = getattr(lib, fn)(*args, ctypes.byref(n))
    return rc, n.value


def test_size_queries(lib):
    B, S, H = 1, 16384, 28
    rc, ws = _sizes(lib, "sage_workspace_size", B, S, H, 128)
    assert rc == OK
    rc, sc = _sizes(lib, "sage_quantize_scratch_size", B, S, H, 128)
    assert rc == OK
    n = ctypes.c_size_t(0)
    assert lib.sage_bundle_size(B, S, H, 128, ctypes.byref(n), None, None) == OK
    # codes: 3 x B*H*S_pad*128 bytes; scales and means are small
    assert n.value >= 7 * B * H * S * 128   # int8/e4m3 codes (3) + fp16 Q/K copies (4)
    assert ws == n.value + sc
    # scratch: a 256-byte work counter, two per-head flag arrays (256-aligned),
    # then fp64 + fp32 per (head, 128-token group, channel), then the fp32
    # reciprocals of each head's 128 V scales
    assert sc == 256 + 2 * 256 + 28 * 128 * 128 * 8 + 28 * 128 * 128 * 4 + 28 * 128 * 4
    # head dimension 64 runs as 14 head pairs of 128 channels, plus each
    # pair's key mean and V scales for the codes items
    rc, sc64 = _sizes(lib, "sage_quantize_scratch_size", B, S, H, 64)
    assert rc == OK
    assert sc64 == 256 + 2 * 256 + 14 * 128 * 128 * 8 + 14 * 128 * 128 * 4 + 14 * 128 * 4 + 14 * 256 * 4
    assert _sizes(lib, "sage_quantize_scratch_size", 1, 1000, 3, 64)[1] == (
        256 + 2 * 256 + 2 * 8 * 128 * 8 + 2 * 8 * 128 * 4 + 2 * 128 * 4 + 2 * 256 * 4)
    assert _sizes(lib, "sage_workspace_size", 1, 100, 2, 96)[0] == HEAD_DIM
    assert _sizes(lib, "sage_workspace_size", 1, 100, 2, 64)[0] == OK
    assert _sizes(lib, "sage_workspace_size", -1, 100, 2, 128)[0] == SHAPE
    assert _sizes(lib, "sage_workspace_size", 1, 2 ** 40, 2, 128)[0] == TOO_LARGE
    assert _sizes(lib, "sage_workspace_size", 0, 0, 0, 128)[0] == OK
    assert lib.sage_workspace_size(1, 1, 1, 128, None) == NULLPTR


def test_bundle_carve_alignment(lib):
    n = ctypes.c_size_t(0)
    c = _lib.Quantized()
    assert lib.sage_bundle_size(2, 1000, 3, 128, ctypes.byref(n), ctypes.c_void_p(0x100000), ctypes.byref(c)) == OK
    ptrs = [c.q_codes_dev, c.k_codes_dev, c.vt_codes_dev, c.q_scale_dev, c.k_scale_dev, c.v_scale_dev, c.k_mean_dev,
            c.q16_dev, c.k16_dev]
    assert ptrs[0] == 0x100000 and all(p % 256 == 0 for p in ptrs)
    assert ptrs == sorted(ptrs) and ptrs[-1] + 2 * 3 * 1024 * 128 * 2 <= 0x100000 + n.value
    assert lib.sage_bundle_size(2, 1000, 3, 128, ctypes.byref(n), ctypes.c_void_p(0x100010), ctypes.byref(c)) == ALIGN


def _call_sageattn(lib, **over):
    a = dict(q=0x10000, k=0x20000, v=0x30000, shape=(1, 256, 2, 128), kshape=None, vshape=None,
             strides=(256 * 2 * 128, 2 * 128, 128, 1), dt=0, kdt=0, vdt=0, layout=b"NHD", causal=0, sm=float("nan"),
             lse=0, smooth=1, out=0x40000, ostrides=None, odt=0, ws=0x50000, wsn=1 << 40)
    a.update(over)
    I = _lib.I64x4
    return lib.sage_sageattn(ctypes.c_void_p(a["q"]), ctypes.c_void_p(a["k"]), ctypes.c_void_p(a["v"]),
                             I(*a["shape"]), I(*(a["kshape"] or a["shape"])), I(*(a["vshape"] or a["shape"])),
                             I(*a["strides"]), I(*a["strides"]), I(*a["strides"]), a["dt"], a["kdt"], a["vdt"],
                             a["layout"], a["causal"], ctypes.c_float(a["sm"]), a["lse"], a["smooth"],
                             ctypes.c_void_p(a["out"]), I(*(a["ostrides"] or a["strides"])), a["odt"],
                             ctypes.c_void_p(a["ws"]), a["wsn"], None)


@pytest.mark.parametrize("over,code", [
    (dict(causal=1), CAUSAL),
    (dict(lse=1), LSE),
    (dict(causal=1, lse=1), CAUSAL),
    (dict(dt=1), DTYPE), (dict(kdt=2), DTYPE), (dict(vdt=3), DTYPE), (dict(odt=1), DTYPE),
    (dict(shape=(1, 256, 2, 64)), HEAD_DIM),
    (dict(kshape=(1, 255, 2, 128)), SHAPE),
    (dict(vshape=(1, 256, 3, 128)), SHAPE),
    (dict(layout=b"BSHD"), LAYOUT),
    (dict(strides=(65536, 256, 128, 2)), LAYOUT),
    (dict(q=0x10008), ALIGN),
    (dict(strides=(65536, 260, 128, 1)), ALIGN),
    (dict(out=0x40004), ALIGN),
    (dict(q=0), NULLPTR), (dict(out=0), NULLPTR), (dict(ws=0), NULLPTR),
    (dict(ws=0x50010), ALIGN),
    (dict(wsn=1000), WORKSPACE),
    (dict(sm=-1.0), ARG), (dict(sm=float("inf")), ARG), (dict(sm=0.0), ARG),
    (dict(shape=(1, 2 ** 40, 2, 128), strides=(2 ** 48, 256, 128, 1)), TOO_LARGE),
])
def test_sageattn_rejections(lib, over, code):
    assert _call_sageattn(lib, **over) == code


def test_quantize_and_attention_rejections(lib):
    t = _lib.Bf16Tensor(0x10000, 65536, 256, 128)
    bad = _lib.Bf16Tensor(0x10002, 65536, 256, 128)
    nul = _lib.Bf16Tensor(0, 65536, 256, 128)
    qz = _lib.Quantized(0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000, 0x700000, 0x800000,
                        0x900000)
    r = ctypes.byref
    assert lib.sage_quantize(r(t), r(t), r(t), 1, 256, 2, 96, 1, r(qz), ctypes.c_void_p(0x800000), 1 << 30, None) == HEAD_DIM
    assert lib.sage_quantize(r(bad), r(t), r(t), 1, 256, 2, 128, 1, r(qz), ctypes.c_void_p(0x800000), 1 << 30, None) == ALIGN
    assert lib.sage_quantize(r(t), r(nul), r(t), 1, 256, 2, 128, 1, r(qz), ctypes.c_void_p(0x800000), 1 << 30, None) == NULLPTR
    assert lib.sage_quantize(r(t), r(t), r(t), 1, 256, 2, 128, 1, r(qz), ctypes.c_void_p(0x800000), 16, None) == WORKSPACE
    assert lib.sage_quantize(r(t), r(t), r(t), 1, 256, 2, 128, 1, r(qz), None, 1 << 30, None) == NULLPTR
    qz_bad = _lib.Quantized(0x100000, 0x200004, 0x300000, 0x400000, 0x500000, 0x600000, 0x700000, 0x800000,
                            0x900000)
    out = ctypes.c_void_p(0x900000)
    plain = lib.sage_attention
    ex = [lambda *a, fn=fn: getattr(lib, fn)(*a[:6], 1, *a[6:10], None, a[10])
          for fn in ("sage_attention_ex", "sage_attention_simt")]
    for f in [plain] + ex:
        assert f(r(qz), 1, 256, 2, 128, ctypes.c_float(-0.1), out, 65536, 256, 128, None) == ARG
        assert f(r(qz), 1, 256, 2, 128, ctypes.c_float(math.nan), out, 65536, 256, 128, None) == ARG
        assert f(r(qz_bad), 1, 256, 2, 128, ctypes.c_float(0.1), out, 65536, 256, 128, None) == ALIGN
        assert f(r(qz), 1, 256, 2, 100, ctypes.c_float(0.1), out, 65536, 256, 128, None) == HEAD_DIM
        assert f(None, 1, 256, 2, 128, ctypes.c_float(0.1), out, 65536, 256, 128, None) == NULLPTR
        assert f(r(qz), 1, 256, 2, 128, ctypes.c_float(0.1), None, 65536, 256, 128, None) == NULLPTR
        assert f(r(qz), 1, 256, 2, 128, ctypes.c_float(0.1), out, 65536, 252, 128, None) == ALIGN
    # a misaligned log-sum-exp buffer
    for fn in ("sage_attention_ex", "sage_attention_simt"):
        assert getattr(lib, fn)(r(qz), 1, 256, 2, 128, ctypes.c_float(0.1), 1, out, 65536, 256, 128,
                                ctypes.c_void_p(0xA00002), None) == ALIGN
    assert lib.sage_lse_smooth_k_term(r(t), ctypes.c_void_p(0x700000), 1, 256, 2, 128, ctypes.c_float(0.1),
                                      ctypes.c_void_p(0xA00002), None) == ALIGN
    assert lib.sage_lse_smooth_k_term(r(t), None, 1, 256, 2, 128, ctypes.c_float(0.1),
                                      ctypes.c_void_p(0xA00000), None) == NULLPTR
    assert lib.sage_lse_smooth_k_term(r(t), ctypes.c_void_p(0x700000), 1, 256, 2, 96, ctypes.c_float(0.1),
                                      ctypes.c_void_p(0xA00000), None) == HEAD_DIM


def test_python_binding_rejects_host_tensors():
    q = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sageattn(q, q, q)
    assert issubclass(SageError, ValueError)


def _call_sageattn_ex(lib, lse_ptr=0x60000, **over):
    a = dict(q=0x10000, k=0x20000, v=0x30000, shape=(1, 256, 2, 128), kshape=None, vshape=None,
             strides=(256 * 2 * 128, 2 * 128, 128, 1), dt=0, kdt=0, vdt=0, layout=b"NHD", causal=1, sm=float("nan"),
             smooth=1, out=0x40000, ostrides=None, odt=0, ws=0x50000, wsn=1 << 40)
    a.update(over)
    I = _lib.I64x4
    return lib.sage_sageattn_ex(ctypes.c_void_p(a["q"]), ctypes.c_void_p(a["k"]), ctypes.c_void_p(a["v"]),
                                I(*a["shape"]), I(*(a["kshape"] or a["shape"])), I(*(a["vshape"] or a["shape"])),
                                I(*a["strides"]), I(*a["strides"]), I(*a["strides"]), a["dt"], a["kdt"], a["vdt"],
                                a["layout"], a["causal"], ctypes.c_float(a["sm"]), a["smooth"],
                                ctypes.c_void_p(a["out"]), I(*(a["ostrides"] or a["strides"])), a["odt"],
                                ctypes.c_void_p(lse_ptr), ctypes.c_void_p(a["ws"]), a["wsn"], None)


@pytest.mark.parametrize("over,code", [
    (dict(dt=1), DTYPE), (dict(odt=1), DTYPE),
    (dict(shape=(1, 256, 2, 96)), HEAD_DIM),
    (dict(kshape=(1, 255, 2, 128)), SHAPE),
    (dict(layout=b"BSHD"), LAYOUT),
    (dict(out=0x40004), ALIGN), (dict(lse_ptr=0x60002), ALIGN),
    (dict(ws=0), NULLPTR), (dict(wsn=1000), WORKSPACE), (dict(sm=-1.0), ARG),
])
def test_sageattn_ex_keeps_the_other_checks(lib, over, code):
    # the extended entry honours is_causal and the log-sum-exp (here both on)
    # and still rejects everything else sage_sageattn rejects
    assert _call_sageattn_ex(lib, **over) == code


def _call_sageattn_host(lib, **over):
    a = dict(q=0x10000, k=0x20000, v=0x30000, shape=(1, 256, 2, 128), dt=0, layout=b"NHD", causal=0,
             sm=float("nan"), smooth=1, out=0x40000, groups=0, ws=0x50000, wsn=1 << 40)
    a.update(over)
    return lib.sage_sageattn_host(ctypes.c_void_p(a["q"]), ctypes.c_void_p(a["k"]), ctypes.c_void_p(a["v"]),
                                  _lib.I64x4(*a["shape"]), a["dt"], a["layout"], a["causal"], ctypes.c_float(a["sm"]),
                                  a["smooth"], ctypes.c_void_p(a["out"]), a["groups"], ctypes.c_void_p(a["ws"]),
                                  a["wsn"], None)


@pytest.mark.parametrize("over,code", [
    (dict(dt=1), DTYPE), (dict(layout=b"BSHD"), LAYOUT), (dict(layout=None), NULLPTR),
    (dict(shape=(1, 256, 2, 96)), HEAD_DIM), (dict(shape=(1, -1, 2, 128)), SHAPE),
    (dict(shape=(1, 1 << 32, 2, 128)), TOO_LARGE), (dict(sm=0.0), ARG), (dict(groups=-1), ARG),
    (dict(q=0), NULLPTR), (dict(out=0), NULLPTR), (dict(ws=0), NULLPTR), (dict(ws=0x50010), ALIGN),
    (dict(wsn=1000), WORKSPACE),
])
def test_sageattn_host_rejections(lib, over, code):
    # every argument check runs on the host before any CUDA call
    assert _call_sageattn_host(lib, **over) == code


def test_sageattn_host_empty_problem_does_nothing(lib):
    assert _call_sageattn_host(lib, shape=(1, 0, 2, 128), q=0, k=0, v=0, out=0, ws=0, wsn=0) == OK
    assert _call_sageattn_host(lib, shape=(0, 256, 2, 128), layout=b"HND") == OK


def test_host_workspace_size_grows_with_groups_in_flight(lib):
    n = ctypes.c_size_t(0)
    assert lib.sage_host_workspace_size(1, 16384, 28, 128, 0, ctypes.byref(n)) == OK
    auto = n.value
    # device copies of q, k, v, out (4 x 117 MB) plus two groups' bundles and scratch
    assert auto >= 4 * 16384 * 28 * 128 * 2
    assert lib.sage_host_workspace_size(1, 16384, 28, 128, 1, ctypes.byref(n)) == OK
    one = n.value  # one group of 28 heads: two full-size bundles
    assert one > auto
    assert lib.sage_host_workspace_size(1, 16384, 28, 128, -1, ctypes.byref(n)) == ARG
    assert lib.sage_host_workspace_size(1, 16384, 28, 96, 0, ctypes.byref(n)) == HEAD_DIM


def test_device_entries_without_a_device_return_an_error(lib):
    # no GPU in this process: the entries that need one report an error
    # code (a failed CUDA call) instead of crashing or launching anything
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    code = ctypes.c_int(0)
    assert lib.sage_selftest_wait_timeout(None) < 0
    assert lib.sage_device_error(None, ctypes.byref(code)) < 0


def _args_struct(lse_ptr=0x60000, **over):
    a = dict(q=0x10000, k=0x20000, v=0x30000, shape=(1, 256, 2, 128), kshape=None, vshape=None,
             strides=(256 * 2 * 128, 2 * 128, 128, 1), dt=0, kdt=0, vdt=0, layout=b"NHD", causal=1, sm=float("nan"),
             smooth=1, out=0x40000, ostrides=None, odt=0, ws=0x50000, wsn=1 << 40)
    a.update(over)
    I = _lib.I64x4
    s = _lib.SageattnArgs()
    s.q_dev, s.k_dev, s.v_dev = a["q"], a["k"], a["v"]
    s.q_shape, s.k_shape, s.v_shape = I(*a["shape"]), I(*(a["kshape"] or a["shape"])), I(*(a["vshape"] or a["shape"]))
    s.q_strides = s.k_strides = s.v_strides = I(*a["strides"])
    s.out_strides = I(*(a["ostrides"] or a["strides"]))
    s.q_dtype, s.k_dtype, s.v_dtype, s.out_dtype = a["dt"], a["kdt"], a["vdt"], a["odt"]
    s.is_causal, s.smooth_k, s.sm_scale = a["causal"], a["smooth"], a["sm"]
    s.tensor_layout = a["layout"]
    s.out_dev, s.lse_dev, s.workspace_dev, s.workspace_bytes = a["out"], lse_ptr, a["ws"], a["wsn"]
    s.cuda_stream = None
    return s


@pytest.mark.parametrize("over,code", [
    (dict(dt=1), DTYPE), (dict(odt=1), DTYPE),
    (dict(shape=(1, 256, 2, 96)), HEAD_DIM),
    (dict(kshape=(1, 255, 2, 128)), SHAPE),
    (dict(layout=b"BSH"), LAYOUT), (dict(layout=b"NHDX"), LAYOUT), (dict(layout=b"NH"), LAYOUT),
    (dict(out=0x40004), ALIGN), (dict(lse_ptr=0x60002), ALIGN), (dict(q=0x10008), ALIGN),
    (dict(ws=0), NULLPTR), (dict(out=0), NULLPTR), (dict(wsn=1000), WORKSPACE), (dict(sm=-1.0), ARG),
    (dict(shape=(1, 2 ** 40, 2, 128), strides=(2 ** 48, 256, 128, 1)), TOO_LARGE),
])
def test_sageattn_args_call_checks_like_the_ex_entry(lib, over, code):
    lse = over.pop("lse_ptr", 0x60000)
    s = _args_struct(lse, **over)
    assert lib.sage_sageattn_args_call(ctypes.byref(s)) == code
    assert _call_sageattn_ex(lib, lse_ptr=lse, **over) == code
    assert lib.sage_sageattn_args_call(None) == NULLPTR


def test_sageattn_args_struct_matches_the_header(tmp_path):
    # the binding's struct must have the C struct's size and field offsets
    # (compiled here with the host compiler from include/sage.h)
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    fields = [f[0] for f in _lib.SageattnArgs._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "sage.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(sage_sageattn_args));\n'
                   + "".join(f'  printf("%zu\\n", offsetof(sage_sageattn_args, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-I", str(_build.ROOT) + "/include", str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got[0] == ctypes.sizeof(_lib.SageattnArgs)
    assert got[1:] == [getattr(_lib.SageattnArgs, f).offset for f in fields]
