"""Thin ctypes binding over libfa.so (include/fa.h). Argument marshalling only.

Every step of attention runs in the library's CUDA kernels; this module only checks
tensor metadata, allocates outputs with torch and passes raw device pointers and the
current CUDA stream. There is no fallback: if libfa.so is missing or the GPU is not an
sm_103 part, calls raise.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK = 0
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float


class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({strerror(status)})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libfa.so once (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m online_softmax_09_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        L.fa_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp]
        L.fa_fwd.restype = _i
        L.fa_fwd_stats.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _vp]
        L.fa_fwd_stats.restype = _i
        L.fa_bwd_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
        L.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.fa_bwd.argtypes = [_vp] * 9 + [_vp, ctypes.c_size_t] + [_i, _i, _i, _i, _i, _i, _f, _vp]
        L.fa_bwd.restype = _i
        L.fa_bwd_noalloc.argtypes = [_vp] * 9 + [_i, _i, _i, _i, _i, _i, _f, _vp]
        L.fa_bwd_noalloc.restype = _i
        L.fa_bwd_window.argtypes = [_vp] * 9 + [_vp, ctypes.c_size_t] + [_i, _i, _i, _i, _i, _i, _f, _vp]
        L.fa_bwd_window.restype = _i
        L.fa_bwd_prepare.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_size_t, _i, _i, _i, _i, _i, _vp]
        L.fa_bwd_prepare.restype = _i
        L.fa_bwd_compute.argtypes = [_vp] * 7 + [ctypes.c_size_t, _i, _i, _i, _i, _i, _i, _f, _vp]
        L.fa_bwd_compute.restype = _i
        L.fa_bwd_finalize.argtypes = [_vp, _vp, ctypes.c_size_t, _i, _i, _i, _i, _i, _f, _vp]
        L.fa_bwd_finalize.restype = _i
        L.fa_fwd_window.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp]
        L.fa_fwd_window.restype = _i
        L.fa_fwd_splitkv_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i]
        L.fa_fwd_splitkv_workspace_bytes.restype = ctypes.c_size_t
        L.fa_fwd_splitkv_auto.argtypes = [_i] * 7
        L.fa_fwd_splitkv_auto.restype = _i
        L.fa_fwd_splitkv.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp,
                                     ctypes.c_size_t, _vp]
        L.fa_fwd_splitkv.restype = _i
        L.fa_naive_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
        L.fa_naive_workspace_bytes.restype = ctypes.c_size_t
        L.fa_naive_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _i, _i, _i, _i, _i, _i, _f, _vp]
        L.fa_naive_fwd.restype = _i
        L.fa_fwd_bwd_host_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
        L.fa_fwd_bwd_host_workspace_bytes.restype = ctypes.c_size_t
        L.fa_fwd_bwd_host.argtypes = [_vp] * 9 + [_i, _i, _i, _i, _i, _i, _f, _vp, ctypes.c_size_t, _vp]
        L.fa_fwd_bwd_host.restype = _i
        L.fa_selftest_wait_timeout.argtypes = [_vp, _vp]
        L.fa_selftest_wait_timeout.restype = _i
        L.fa_softmax_rows.argtypes = [_vp, _vp, _vp, ctypes.c_longlong, _i, _vp]
        L.fa_softmax_rows.restype = _i
        L.fa_check.argtypes = [_vp]
        L.fa_check.restype = _i
        L.fa_strerror.argtypes = [_i]
        L.fa_strerror.restype = ctypes.c_char_p
        L.fa_version.argtypes = []
        L.fa_version.restype = _i
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().fa_strerror(int(status)).decode()


def _stream_handle(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def _check_qkv(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D bfloat16 CUDA tensor [B, H, N, d]")
    B, Hq, N, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError("k and v must be [B, Hkv, N, d] with the same B, N, d as q")
    return B, Hq, k.shape[1], N, d


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
            stream=None, counters=None):
    """O, LSE = attention(q, k, v). q [B,Hq,N,d], k/v [B,Hkv,N,d] bf16 CUDA tensors."""
    B, Hq, Hkv, N, d = _check_qkv(q, k, v)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    sc = 0.0 if scale is None else float(scale)
    h = _stream_handle(stream, q.device)
    if counters is None:
        r = lib().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                         B, Hq, Hkv, N, d, int(bool(causal)), sc, h)
    else:
        r = lib().fa_fwd_stats(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                               B, Hq, Hkv, N, d, int(bool(causal)), sc, counters.data_ptr(), h)
    if r != FA_OK:
        raise FAError(r, "fa_fwd")
    return o, l


def forward_window(q, k, v, window: int, scale: float | None = None, out=None, lse=None, stream=None):
    """Causal sliding-window attention (fa_fwd_window): query i sees keys i-window < j <= i."""
    B, Hq, Hkv, N, d = _check_qkv(q, k, v)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    sc = 0.0 if scale is None else float(scale)
    r = lib().fa_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                            B, Hq, Hkv, N, d, int(window), sc, _stream_handle(stream, q.device))
    if r != FA_OK:
        raise FAError(r, "fa_fwd_window")
    return o, l


def forward_splitkv(q, k, v, causal: bool = False, num_splits: int = 0, scale: float | None = None,
                    out=None, lse=None, workspace=None, stream=None):
    """Split-KV forward (fa_fwd_splitkv); num_splits <= 0 lets the library choose."""
    B, Hq, Hkv, N, d = _check_qkv(q, k, v)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    if workspace is None:
        used = int(num_splits) if num_splits > 0 else splitkv_auto(
            B, Hq, Hkv, N, d, causal, torch.cuda.get_device_properties(q.device).multi_processor_count)
        n = int(lib().fa_fwd_splitkv_workspace_bytes(B, Hq, Hkv, N, d, used))
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    sc = 0.0 if scale is None else float(scale)
    r = lib().fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                             B, Hq, Hkv, N, d, int(bool(causal)), sc, int(num_splits), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    if r != FA_OK:
        raise FAError(r, "fa_fwd_splitkv")
    return o, l


def splitkv_auto(B: int, Hq: int, Hkv: int, N: int, d: int, causal: bool, num_sms: int) -> int:
    """The split count fa_fwd_splitkv picks for num_splits <= 0 on a GPU with num_sms SMs."""
    r = lib().fa_fwd_splitkv_auto(B, Hq, Hkv, N, d, int(bool(causal)), num_sms)
    if r < 0:
        raise FAError(r, "fa_fwd_splitkv_auto")
    return r


def forward_naive(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, workspace=None,
                  stream=None):
    """Baseline standard attention with S and P in HBM (fa_naive_fwd)."""
    B, Hq, Hkv, N, d = _check_qkv(q, k, v)
    o = out if out is not None else torch.empty_like(q)
    l = lse if lse is not None else torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(int(lib().fa_naive_workspace_bytes(B, Hq, Hkv, N, d)), dtype=torch.uint8,
                                device=q.device)
    sc = 0.0 if scale is None else float(scale)
    r = lib().fa_naive_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(), workspace.data_ptr(),
                           workspace.numel() * workspace.element_size(), B, Hq, Hkv, N, d, int(bool(causal)), sc,
                           _stream_handle(stream, q.device))
    if r != FA_OK:
        raise FAError(r, "fa_naive_fwd")
    return o, l


def workspace_bytes(B: int, Hq: int, Hkv: int, N: int, d: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, Hq, Hkv, N, d))


def backward(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV of attention given the forward's o and lse and the output gradient do."""
    B, Hq, Hkv, N, d = _check_qkv(q, k, v)
    for name, t in (("o", o), ("do", do)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must match q")
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(k)
    dv = dv if dv is not None else torch.empty_like(v)
    nbytes = workspace_bytes(B, Hq, Hkv, N, d)
    ws = workspace if workspace is not None else torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    sc = 0.0 if scale is None else float(scale)
    r = lib().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                     dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(),
                     B, Hq, Hkv, N, d, int(bool(causal)), sc, _stream_handle(stream, q.device))
    if r != FA_OK:
        raise FAError(r, "fa_bwd")
    return dq, dk, dv


def backward_noalloc(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
                     dq=None, dk=None, dv=None, stream=None):
    """fa_bwd_noalloc: the backward without a caller workspace (the library's fixed scratch
    array; calls that overlap on one device race on it)."""
    B, Hq, Hkv, N, d = _check_qkv(q, k, v)
    for name, t in (("o", o), ("do", do)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must match q")
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(k)
    dv = dv if dv is not None else torch.empty_like(v)
    sc = 0.0 if scale is None else float(scale)
    r = lib().fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                             dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, d, int(bool(causal)), sc,
                             _stream_handle(stream, q.device))
    if r != FA_OK:
        raise FAError(r, "fa_bwd_noalloc")
    return dq, dk, dv


def backward_window(q, k, v, o, do, lse, window: int, scale: float | None = None,
                    dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients of causal sliding-window attention (fa_bwd_window)."""
    B, Hq, Hkv, N, d = _check_qkv(q, k, v)
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(k)
    dv = dv if dv is not None else torch.empty_like(v)
    ws = workspace if workspace is not None else torch.empty(workspace_bytes(B, Hq, Hkv, N, d), dtype=torch.uint8,
                                                              device=q.device)
    sc = 0.0 if scale is None else float(scale)
    r = lib().fa_bwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                            ws.numel() * ws.element_size(), B, Hq, Hkv, N, d, int(window), sc,
                            _stream_handle(stream, q.device))
    if r != FA_OK:
        raise FAError(r, "fa_bwd_window")
    return dq, dk, dv


def backward_stages(q, k, v, o, do, lse, dq, dk, dv, workspace, causal: bool = False,
                    scale: float | None = None, stream=None, between=None, only=None):
    """Run fa_bwd_prepare, fa_bwd_compute and fa_bwd_finalize; ``between(i)`` (optional)
    is called before stage i (0, 1, 2) and after the last (3), e.g. to record CUDA events.
    ``only`` (optional): the stage indices to run, e.g. ``(1,)`` for the compute stage alone on a
    workspace an earlier prepare filled."""
    B, Hq, Hkv, N, d = _check_qkv(q, k, v)
    sc = 0.0 if scale is None else float(scale)
    h = _stream_handle(stream, q.device)
    nb = workspace.numel() * workspace.element_size()
    L = lib()
    calls = (
        lambda: L.fa_bwd_prepare(o.data_ptr(), do.data_ptr(), lse.data_ptr(), workspace.data_ptr(), nb,
                                 B, Hq, Hkv, N, d, h),
        lambda: L.fa_bwd_compute(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), workspace.data_ptr(), nb, B, Hq, Hkv, N, d, int(bool(causal)), sc, h),
        lambda: L.fa_bwd_finalize(dq.data_ptr(), workspace.data_ptr(), nb, B, Hq, Hkv, N, d, sc, h),
    )
    for i, call in enumerate(calls):
        if only is not None and i not in only:
            continue
        if between is not None:
            between(i)
        r = call()
        if r != FA_OK:
            raise FAError(r, ("fa_bwd_prepare", "fa_bwd_compute", "fa_bwd_finalize")[i])
    if between is not None:
        between(3)
    return dq, dk, dv


def fwd_bwd_host_workspace_bytes(B: int, Hq: int, Hkv: int, N: int, d: int) -> int:
    """Device workspace bytes for fa_fwd_bwd_host."""
    n = lib().fa_fwd_bwd_host_workspace_bytes(B, Hq, Hkv, N, d)
    if n == 0:
        raise ValueError("invalid sizes")
    return n


def fwd_bwd_host(q, k, v, do, causal: bool = False, scale: float | None = None, out=None, workspace=None,
                 device=None, stream=None):
    """Forward and backward on host (CPU, ideally pinned) bf16 tensors (fa_fwd_bwd_host).

    Returns host tensors ``(o, lse, dq, dk, dv)``; ``out`` may supply them (o, dq, dk, dv bf16
    and lse fp32, contiguous CPU tensors). ``workspace`` is a CUDA uint8 tensor of at least
    fwd_bwd_host_workspace_bytes(...) bytes (allocated when None). Asynchronous: the outputs
    are ready after the stream is synchronised (e.g. check())."""
    for name, t in (("q", q), ("k", k), ("v", v), ("do", do)):
        if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D bfloat16 CPU tensor [B, H, N, d]")
    B, Hq, N, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != N or k.shape[3] != d or do.shape != q.shape:
        raise ValueError("k, v must be [B, Hkv, N, d] and do [B, Hq, N, d] with the same B, N, d as q")
    Hkv = k.shape[1]
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    if out is None:
        pin = q.is_pinned()
        out = (torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin),
               torch.empty((B, Hq, N), dtype=torch.float32, pin_memory=pin),
               torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin),
               torch.empty(k.shape, dtype=torch.bfloat16, pin_memory=pin),
               torch.empty(k.shape, dtype=torch.bfloat16, pin_memory=pin))
    o, lse, dq, dk, dv = out
    for t, shape, dt in ((o, q.shape, torch.bfloat16), (lse, (B, Hq, N), torch.float32), (dq, q.shape, torch.bfloat16),
                         (dk, k.shape, torch.bfloat16), (dv, k.shape, torch.bfloat16)):
        if t.is_cuda or tuple(t.shape) != tuple(shape) or t.dtype != dt or not t.is_contiguous():
            raise ValueError("out must be contiguous CPU tensors (o, lse, dq, dk, dv) of the input shapes")
    nbytes = fwd_bwd_host_workspace_bytes(B, Hq, Hkv, N, d)
    ws = workspace if workspace is not None else torch.empty(nbytes, dtype=torch.uint8, device=dev)
    sc = 0.0 if scale is None else float(scale)
    r = lib().fa_fwd_bwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, d, int(bool(causal)), sc,
                              ws.data_ptr(), ws.numel() * ws.element_size(), _stream_handle(stream, dev))
    if r != FA_OK:
        raise FAError(r, "fa_fwd_bwd_host")
    return o, lse, dq, dk, dv


def selftest_wait_timeout(device=None, stream=None) -> int:
    """Run fa_selftest_wait_timeout: one warp waits on a barrier nothing completes until the
    bounded wait gives up (2 s). Returns the kernel's result code (2: gave up and raised its
    abort flag); the device status then holds the timeout, which check() reports."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    res = torch.zeros(1, dtype=torch.int32, device=dev)
    r = lib().fa_selftest_wait_timeout(res.data_ptr(), _stream_handle(stream, dev))
    if r != FA_OK:
        raise FAError(r, "fa_selftest_wait_timeout")
    (stream if stream is not None else torch.cuda.current_stream(dev)).synchronize()
    return int(res.item())


def softmax_rows(x, out=None, lse=None, with_lse: bool = True, stream=None):
    """Row-wise online softmax of a contiguous fp32 CUDA tensor [..., n] (fa_softmax_rows)."""
    if not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    n = x.shape[-1]
    rows = x.numel() // n
    p = out if out is not None else torch.empty_like(x)
    l = lse if lse is not None else (torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
                                     if with_lse else None)
    r = lib().fa_softmax_rows(x.data_ptr(), p.data_ptr(), l.data_ptr() if l is not None else None, rows, n,
                              _stream_handle(stream, x.device))
    if r != FA_OK:
        raise FAError(r, "fa_softmax_rows")
    return p, l


def check(stream=None, device=None) -> None:
    """Synchronise the stream and raise if a kernel reported a device-side failure."""
    dev = device if device is not None else torch.cuda.current_device()
    r = lib().fa_check(_stream_handle(stream, dev))
    if r != FA_OK:
        raise FAError(r, "fa_check")


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
