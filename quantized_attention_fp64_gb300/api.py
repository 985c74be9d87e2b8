"""Python entry points over the C ABI (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; PyTorch is
used here only to allocate device buffers and to name the current stream.
If the library is missing the calls raise; there is no other code path.
"""

from __future__ import annotations

import ctypes
import math
import threading
from dataclasses import dataclass

import torch

from . import _lib

SAGE_ERR_SHAPE = -5
SAGE_ERR_LAYOUT = -6

_DTYPE_CODES = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}


class SageError(ValueError):
    """A call rejected by the library; ``code`` is the SAGE_ERR_* value."""

    def __init__(self, code: int, message: str):
        super().__init__(f"{message} (sage error {code})")
        self.code = code


def _check(rc: int) -> None:
    if rc != 0:
        raise SageError(rc, _lib.load().sage_strerror(rc).decode())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    return _DTYPE_CODES.get(t.dtype, 3)


def _bsh(shape, layout: str):
    """(B, S, H, D) from a shape given in ``layout`` order."""
    if layout == "HND":
        return shape[0], shape[2], shape[1], shape[3]
    return shape[0], shape[1], shape[2], shape[3]


def _bsh_strides(t: torch.Tensor, layout: str):
    st = t.stride()
    if layout == "HND":
        return st[0], st[2], st[1]
    return st[0], st[1], st[2]


def workspace_size(B: int, S: int, H: int, D: int = 128) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.load().sage_workspace_size(B, S, H, D, ctypes.byref(n)))
    return n.value


def quantize_scratch_size(B: int, S: int, H: int, D: int = 128) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.load().sage_quantize_scratch_size(B, S, H, D, ctypes.byref(n)))
    return n.value


@dataclass
class QuantizedQKV:
    """Quantized bundle (views into one device buffer, see sage_quantized)."""

    buffer: torch.Tensor
    q_codes: torch.Tensor   # int8 [B, H, S_pad, D]
    k_codes: torch.Tensor   # int8 [B, H, S_pad, D]
    vt_codes: torch.Tensor  # uint8 (e4m3fn) [B, H, D, S_pad]
    q_scale: torch.Tensor   # float32 [B, H, S_pad/32]
    k_scale: torch.Tensor   # float32 [B, H, S_pad/32]
    v_scale: torch.Tensor   # float32 [B, H, D]
    k_mean: torch.Tensor    # float32 [B, H, D]
    q16: torch.Tensor       # float16 [B, H, S_pad, D], the Q codes as fp16 values
    k16: torch.Tensor       # float16 [B, H, S_pad, D], the K codes as fp16 values
    B: int
    S: int
    H: int
    D: int = 128

    def c_struct(self) -> _lib.Quantized:
        return _lib.Quantized(*(t.data_ptr() for t in (self.q_codes, self.k_codes, self.vt_codes, self.q_scale,
                                                       self.k_scale, self.v_scale, self.k_mean, self.q16,
                                                       self.k16)))


def alloc_bundle(B: int, S: int, H: int, device, D: int = 128) -> QuantizedQKV:
    lib = _lib.load()
    n = ctypes.c_size_t(0)
    _check(lib.sage_bundle_size(B, S, H, D, ctypes.byref(n), None, None))
    buf = torch.empty(max(n.value, 256), dtype=torch.uint8, device=device)
    c = _lib.Quantized()
    _check(lib.sage_bundle_size(B, S, H, D, ctypes.byref(n), ctypes.c_void_p(buf.data_ptr()), ctypes.byref(c)))
    s_pad = -(-S // 128) * 128
    base = buf.data_ptr()

    def view(ptr, dtype, shape):
        off = ptr - base
        count = 1
        for x in shape:
            count *= x
        nbytes = count * torch.tensor([], dtype=dtype).element_size()
        return buf[off:off + nbytes].view(dtype).view(shape)

    return QuantizedQKV(
        buffer=buf,
        q_codes=view(c.q_codes_dev, torch.int8, (B, H, s_pad, D)),
        k_codes=view(c.k_codes_dev, torch.int8, (B, H, s_pad, D)),
        vt_codes=view(c.vt_codes_dev, torch.uint8, (B, H, D, s_pad)),
        q_scale=view(c.q_scale_dev, torch.float32, (B, H, s_pad // 32)),
        k_scale=view(c.k_scale_dev, torch.float32, (B, H, s_pad // 32)),
        v_scale=view(c.v_scale_dev, torch.float32, (B, H, D)),
        k_mean=view(c.k_mean_dev, torch.float32, (B, H, D)),
        q16=view(c.q16_dev, torch.float16, (B, H, s_pad, D)),
        k16=view(c.k16_dev, torch.float16, (B, H, s_pad, D)),
        B=B, S=S, H=H, D=D)


def _bf16_tensor(t: torch.Tensor, layout: str) -> _lib.Bf16Tensor:
    sb, ss, sh = _bsh_strides(t, layout)
    return _lib.Bf16Tensor(t.data_ptr(), sb, ss, sh)


def _require_cuda(*ts):
    for t in ts:
        if not isinstance(t, torch.Tensor):
            raise TypeError("expected torch tensors")
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")


def quantize(q, k, v, tensor_layout: str = "NHD", smooth_k: bool = True, out: QuantizedQKV | None = None,
             scratch: torch.Tensor | None = None) -> QuantizedQKV:
    """The quantization prologue (sage_quantize) on BF16 tensors."""
    _require_cuda(q, k, v)
    if q.dim() != 4 or tuple(q.shape) != tuple(k.shape) or tuple(q.shape) != tuple(v.shape):
        raise SageError(SAGE_ERR_SHAPE, "q, k and v must have identical 4-d shapes")
    if tensor_layout not in ("NHD", "HND"):
        raise SageError(SAGE_ERR_LAYOUT, "tensor_layout must be NHD or HND")
    if q.stride(3) != 1 or k.stride(3) != 1 or v.stride(3) != 1:
        raise SageError(SAGE_ERR_LAYOUT, "the channel stride must be 1")
    B, S, H, D = _bsh(q.shape, tensor_layout)
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise SageError(-3, "inputs and output must be bfloat16")
    lib = _lib.load()
    with torch.cuda.device(q.device):
        qz = out if out is not None else alloc_bundle(B, S, H, q.device, D)
        if scratch is None:
            scratch = torch.empty(max(quantize_scratch_size(B, S, H, D), 256), dtype=torch.uint8, device=q.device)
        bundle = qz.c_struct()
        _check(lib.sage_quantize(ctypes.byref(_bf16_tensor(q, tensor_layout)), ctypes.byref(_bf16_tensor(k, tensor_layout)),
                                 ctypes.byref(_bf16_tensor(v, tensor_layout)), B, S, H, D, int(bool(smooth_k)),
                                 ctypes.byref(bundle), ctypes.c_void_p(scratch.data_ptr()), scratch.numel(),
                                 _stream(q.device)))
    return qz


def _attention(fn_name: str, qz: QuantizedQKV, sm_scale, tensor_layout: str, out, is_causal=False,
               return_lse=False):
    lib = _lib.load()
    B, S, H, D = qz.B, qz.S, qz.H, qz.D
    device = qz.buffer.device
    if out is None:
        shape = (B, H, S, D) if tensor_layout == "HND" else (B, S, H, D)
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    scale = (1.0 / math.sqrt(D)) if sm_scale is None else float(sm_scale)
    ob, os_, oh = _bsh_strides(out, tensor_layout)
    bundle = qz.c_struct()
    lse = torch.empty((B, H, S), dtype=torch.float32, device=device) if return_lse else None
    with torch.cuda.device(device):
        if fn_name == "sage_attention":
            _check(lib.sage_attention(ctypes.byref(bundle), B, S, H, D, ctypes.c_float(scale),
                                      ctypes.c_void_p(out.data_ptr()), ob, os_, oh, _stream(device)))
        else:
            _check(getattr(lib, fn_name)(ctypes.byref(bundle), B, S, H, D, ctypes.c_float(scale),
                                         int(bool(is_causal)), ctypes.c_void_p(out.data_ptr()), ob, os_, oh,
                                         ctypes.c_void_p(lse.data_ptr() if lse is not None else None),
                                         _stream(device)))
    return (out, lse) if return_lse else out


def attention(qz: QuantizedQKV, sm_scale=None, tensor_layout: str = "NHD", out=None, is_causal: bool = False,
              return_lse: bool = False):
    """Tensor-core attention on a quantized bundle: sage_attention, or
    sage_attention_ex when a causal mask or the log-sum-exp is asked for
    (then it returns (out, lse) with lse fp32 [B, H, S], the log-sum-exp of
    the bundle's logits; see lse_smooth_k_term)."""
    if not is_causal and not return_lse:
        return _attention("sage_attention", qz, sm_scale, tensor_layout, out)
    return _attention("sage_attention_ex", qz, sm_scale, tensor_layout, out, is_causal, return_lse)


def attention_simt(qz: QuantizedQKV, sm_scale=None, tensor_layout: str = "NHD", out=None, is_causal: bool = False,
                   return_lse: bool = False):
    """The SIMT cross-check kernel (sage_attention_simt); for tests."""
    return _attention("sage_attention_simt", qz, sm_scale, tensor_layout, out, is_causal, return_lse)


def lse_smooth_k_term(q: torch.Tensor, qz: QuantizedQKV, lse: torch.Tensor, sm_scale=None,
                      tensor_layout: str = "NHD") -> torch.Tensor:
    """Adds sm_scale * q_i . k_mean to lse in place (sage_lse_smooth_k_term):
    the log-sum-exp of the mean-reduced keys becomes that of the original keys."""
    _require_cuda(q)
    lib = _lib.load()
    scale = (1.0 / math.sqrt(qz.D)) if sm_scale is None else float(sm_scale)
    with torch.cuda.device(q.device):
        _check(lib.sage_lse_smooth_k_term(ctypes.byref(_bf16_tensor(q, tensor_layout)),
                                          ctypes.c_void_p(qz.k_mean.data_ptr()), qz.B, qz.S, qz.H, qz.D,
                                          ctypes.c_float(scale), ctypes.c_void_p(lse.data_ptr()), _stream(q.device)))
    return lse


# Per-call host work matters for short calls, so the sageattn entries keep it
# small: shape and stride arrays are reused, the workspace of calls up to
# _WS_CACHE_MAX bytes is kept per (thread, device, stream) and reused by the
# thread's next call on that stream, and the stream is read as a raw handle.
# Reuse is safe in stream order within one thread; two threads on one stream
# get separate workspaces, since the library call releases the GIL and their
# launches (prologue, attention) may interleave on the stream.
_WS_CACHE_MAX = 256 << 20
_tls = threading.local()
_i64_cache: dict = {}
_ws_size_cache: dict = {}
_LAYOUTS = {"NHD": b"NHD", "HND": b"HND"}
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(index: int) -> int:
    if _raw_stream is not None:
        return _raw_stream(index)
    return torch.cuda.current_stream(index).cuda_stream


def _i64x4(t) -> "_lib.I64x4":
    arr = _i64_cache.get(t)
    if arr is None:
        if len(_i64_cache) > 512:
            _i64_cache.clear()
        arr = _i64_cache[t] = _lib.I64x4(*t)
    return arr


def _ws_bytes(lib, B, S, H, D):
    key = (B, S, H, D)
    n = _ws_size_cache.get(key)
    if n is None:
        c = ctypes.c_size_t(0)
        n = c.value if lib.sage_workspace_size(B, S, H, D, ctypes.byref(c)) == 0 else -1
        if len(_ws_size_cache) > 512:
            _ws_size_cache.clear()
        _ws_size_cache[key] = n
    return n


def _workspace(device, stream: int, nbytes: int) -> torch.Tensor:
    if nbytes > _WS_CACHE_MAX:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    cache = getattr(_tls, "ws", None)
    if cache is None:
        cache = _tls.ws = {}
    key = (device.index, stream)
    ws = cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        cache[key] = ws
    return ws


def release_workspace_cache() -> None:
    """Drops the workspaces this thread keeps for short sageattn calls."""
    _tls.ws = {}


# Calls whose shapes, strides, dtypes, devices, layout and flags were seen
# before on this thread skip the checks and conversions: the thread keeps one
# filled sage_sageattn_args per signature and changes only the pointers,
# sm_scale and the stream (short calls spend a noticeable share of their time
# in argument marshalling). Per thread, so that no other thread rewrites a
# struct while the library reads it.
_get_device = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device
_NAN = float("nan")


def _call_key(ex, q, k, v, tensor_layout, is_causal, smooth_k):
    return (ex, q.shape, q.stride(), k.shape, k.stride(), v.shape, v.stride(), q.dtype, k.dtype, v.dtype,
            q.get_device(), k.get_device(), v.get_device(), tensor_layout, bool(is_causal), bool(smooth_k))


def _sageattn_fast(ex: bool, q, k, v, tensor_layout, is_causal, sm_scale, return_lse, smooth_k, out, workspace):
    """The call from kept arguments, or None when this thread has not seen the
    signature (or the call needs the full path: a given out or workspace, or
    the LSE)."""
    if out is not None or workspace is not None or return_lse:
        return None
    cache = getattr(_tls, "calls", None)
    if not cache:
        return None
    try:
        prep = cache.get(_call_key(ex, q, k, v, tensor_layout, is_causal, smooth_k))
    except (AttributeError, TypeError):
        return None
    if prep is None:
        return None
    args, ref, fn, device, shape, contiguous, ws_n = prep
    if device.index != _get_device():
        return None
    stream = _stream_handle(device.index)
    out = torch.empty_like(q) if contiguous else torch.empty(shape, dtype=torch.bfloat16, device=device)
    ws = _workspace(device, stream, ws_n)
    args.q_dev = q.data_ptr()
    args.k_dev = k.data_ptr()
    args.v_dev = v.data_ptr()
    args.out_dev = out.data_ptr()
    args.workspace_dev = ws.data_ptr()
    args.workspace_bytes = ws.numel()
    args.cuda_stream = stream
    args.sm_scale = _NAN if sm_scale is None else float(sm_scale)
    _check(fn(ref))
    return out


def _forget_calls() -> dict:
    """Drops this thread's kept call arguments; returns the dict now in use."""
    _tls.calls = {}
    return _tls.calls


def _remember(ex, q, k, v, tensor_layout, is_causal, smooth_k, lib, shape, ws_n, out):
    """Keeps the arguments of a successful call for its signature (this thread)."""
    cache = getattr(_tls, "calls", None)
    if cache is None or len(cache) > 256:
        cache = _tls.calls = {}
    a = _lib.SageattnArgs()
    a.q_shape, a.k_shape, a.v_shape = _lib.I64x4(*q.shape), _lib.I64x4(*k.shape), _lib.I64x4(*v.shape)
    a.q_strides, a.k_strides, a.v_strides = _lib.I64x4(*q.stride()), _lib.I64x4(*k.stride()), _lib.I64x4(*v.stride())
    a.out_strides = _lib.I64x4(*out.stride())
    a.q_dtype, a.k_dtype, a.v_dtype, a.out_dtype = _dtype_code(q), _dtype_code(k), _dtype_code(v), _dtype_code(out)
    a.is_causal, a.smooth_k = int(bool(is_causal)), int(bool(smooth_k))
    a.tensor_layout = tensor_layout.encode()
    a.lse_dev = None
    contiguous = q.is_contiguous() and tuple(out.stride()) == tuple(q.stride())
    cache[_call_key(ex, q, k, v, tensor_layout, is_causal, smooth_k)] = (
        a, ctypes.byref(a), lib.sage_sageattn_args_call, q.device, shape, contiguous, ws_n)


def _sageattn_call(ex: bool, q, k, v, tensor_layout, is_causal, sm_scale, return_lse, smooth_k, out, workspace):
    fast = _sageattn_fast(ex, q, k, v, tensor_layout, is_causal, sm_scale, return_lse, smooth_k, out, workspace)
    if fast is not None:
        return fast
    given_out, given_ws = out is not None, workspace is not None
    for t in (q, k, v):
        if not isinstance(t, torch.Tensor):
            raise TypeError("expected torch tensors")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("tensors must live on a CUDA device")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise SageError(SAGE_ERR_SHAPE, "q, k and v must be 4-d")
    lib = _lib.load()
    layout = tensor_layout if isinstance(tensor_layout, str) else str(tensor_layout)
    shape = tuple(q.shape)
    B, S, H, D = _bsh(shape, layout)
    ws_n = _ws_bytes(lib, B, S, H, D)
    proceed = (ws_n >= 0 and layout in _LAYOUTS and q.dtype == k.dtype == v.dtype == torch.bfloat16
               and shape == tuple(k.shape) == tuple(v.shape) and (ex or not (is_causal or return_lse)))
    device = q.device
    index = device.index
    switch = index != torch.cuda.current_device()
    ctx = torch.cuda.device(device) if switch else None
    if ctx is not None:
        ctx.__enter__()
    try:
        stream = _stream_handle(index)
        lse = None
        if proceed:
            if out is None:
                out = torch.empty(shape, dtype=torch.bfloat16, device=device)
            if workspace is None or workspace.numel() < ws_n:
                workspace = _workspace(device, stream, ws_n)
            if ex and return_lse:
                lse = torch.empty((B, H, S), dtype=torch.float32, device=device)
        out_ptr = out.data_ptr() if out is not None else None
        out_strides = _i64x4(out.stride()) if out is not None else _i64x4((0, 0, 0, 1))
        out_dtype = _dtype_code(out) if out is not None else 0
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_size = workspace.numel() if workspace is not None else 0
        scale = float("nan") if sm_scale is None else float(sm_scale)
        qs, ks, vs = _i64x4(shape), _i64x4(tuple(k.shape)), _i64x4(tuple(v.shape))
        qst, kst, vst = _i64x4(q.stride()), _i64x4(k.stride()), _i64x4(v.stride())
        lay = _LAYOUTS.get(layout) or layout.encode()
        dq, dk, dv = _dtype_code(q), _dtype_code(k), _dtype_code(v)
        if ex:
            rc = lib.sage_sageattn_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), qs, ks, vs, qst, kst, vst, dq, dk, dv,
                                      lay, int(bool(is_causal)), scale, int(bool(smooth_k)), out_ptr, out_strides,
                                      out_dtype, lse.data_ptr() if lse is not None else None, ws_ptr, ws_size,
                                      stream)
        else:
            rc = lib.sage_sageattn(q.data_ptr(), k.data_ptr(), v.data_ptr(), qs, ks, vs, qst, kst, vst, dq, dk, dv,
                                   lay, int(bool(is_causal)), scale, int(bool(return_lse)), int(bool(smooth_k)),
                                   out_ptr, out_strides, out_dtype, ws_ptr, ws_size, stream)
    finally:
        if ctx is not None:
            ctx.__exit__(None, None, None)
    _check(rc)
    if (not (given_out or given_ws or return_lse) and out is not None and out.is_contiguous()
            and layout in _LAYOUTS and not (is_causal and not ex)):
        _remember(ex, q, k, v, layout, is_causal, smooth_k, lib, shape, ws_n, out)
    return (out, lse) if (ex and return_lse) else out


def sageattn(q, k, v, tensor_layout: str = "NHD", is_causal: bool = False, sm_scale=None,
             return_lse: bool = False, smooth_k: bool = True, out=None, workspace=None) -> torch.Tensor:
    """sageattn(q, k, v, tensor_layout, is_causal, sm_scale, return_lse) through sage_sageattn.

    Unsupported inputs (causal, LSE, non-BF16, head dim != 128, unequal
    shapes, unknown layout) raise SageError; nothing falls back.
    """
    return _sageattn_call(False, q, k, v, tensor_layout, is_causal, sm_scale, return_lse, smooth_k, out, workspace)


def sageattn_ex(q, k, v, tensor_layout: str = "NHD", is_causal: bool = False, sm_scale=None,
                return_lse: bool = False, smooth_k: bool = True, out=None, workspace=None):
    """sageattn with is_causal and return_lse honoured (sage_sageattn_ex):
    returns out, or (out, lse) with lse fp32 [B, H, S], the natural-log
    log-sum-exp of each query row's scaled logits. Other unsupported inputs
    raise SageError as in sageattn."""
    return _sageattn_call(True, q, k, v, tensor_layout, is_causal, sm_scale, return_lse, smooth_k, out, workspace)


def host_workspace_size(B: int, S: int, H: int, D: int = 128, n_groups: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.load().sage_host_workspace_size(B, S, H, D, n_groups, ctypes.byref(n)))
    return n.value


def sageattn_host(q, k, v, tensor_layout: str = "NHD", is_causal: bool = False, sm_scale=None,
                  smooth_k: bool = True, out=None, workspace=None, n_groups: int = 0, device=None):
    """sageattn on host (CPU) tensors through sage_sageattn_host: the head
    groups' copies to and from the GPU overlap the kernels of the other
    groups. q, k, v: contiguous BF16 CPU tensors (pinned memory lets the
    copies run asynchronously). Returns out, a CPU tensor (pinned when q is),
    written asynchronously: synchronize the current CUDA stream before
    reading it. The work runs on ``device`` (default: the current CUDA device)."""
    for t in (q, k, v):
        if not isinstance(t, torch.Tensor):
            raise TypeError("expected torch tensors")
        if t.is_cuda:
            raise ValueError("sageattn_host takes host (CPU) tensors; use sageattn for device tensors")
        if not t.is_contiguous():
            raise SageError(SAGE_ERR_LAYOUT, "host tensors must be contiguous")
    if q.dim() != 4 or tuple(q.shape) != tuple(k.shape) or tuple(q.shape) != tuple(v.shape):
        raise SageError(SAGE_ERR_SHAPE, "q, k and v must have identical 4-d shapes")
    lib = _lib.load()
    layout = tensor_layout if isinstance(tensor_layout, str) else str(tensor_layout)
    B, S, H, D = _bsh(tuple(q.shape), layout)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=q.is_pinned())
    elif out.is_cuda or not out.is_contiguous() or tuple(out.shape) != tuple(q.shape):
        raise SageError(SAGE_ERR_SHAPE, "out must be a contiguous host tensor of q's shape")
    with torch.cuda.device(dev):
        n = ctypes.c_size_t(0)
        rc = lib.sage_host_workspace_size(B, S, H, D, n_groups, ctypes.byref(n))
        if rc == 0 and (workspace is None or workspace.numel() < n.value):
            workspace = torch.empty(max(n.value, 256), dtype=torch.uint8, device=dev)
        scale = float("nan") if sm_scale is None else float(sm_scale)
        rc = lib.sage_sageattn_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), _i64x4(tuple(q.shape)), _dtype_code(q),
                                    _LAYOUTS.get(layout) or layout.encode(), int(bool(is_causal)), scale,
                                    int(bool(smooth_k)), out.data_ptr(), int(n_groups),
                                    workspace.data_ptr() if workspace is not None else None,
                                    workspace.numel() if workspace is not None else 0, _stream_handle(dev.index))
    _check(rc)
    return out


def device_error(device=None) -> int:
    """Synchronizes the current stream and returns (and clears) the device error word."""
    lib = _lib.load()
    code = ctypes.c_int(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib.sage_device_error(_stream(dev), ctypes.byref(code)))
    return code.value
