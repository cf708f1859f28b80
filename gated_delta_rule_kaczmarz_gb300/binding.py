"""Thin Python binding of the C ABI in include/kla.h (ctypes).

Argument marshalling only: every step of the computation runs in the CUDA
library ``libkla_gb300.so``.  PyTorch provides device memory and streams.
There is no CPU fallback: if the library cannot be loaded, every call raises.

The functions carry the C names.  Tensor arguments are torch tensors on one
CUDA device, contiguous, in the layouts that kla.h documents; outputs and the
workspace are allocated with torch when not supplied.  A non-OK status raises
``KlaError`` with the library's own message.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

KLA_OK = 0
KLA_ERR_INVALID_ARG = 1
KLA_ERR_UNSUPPORTED = 2
KLA_ERR_CUDA = 3
KLA_ERR_TIMEOUT = 4
KLA_ERR_WORKSPACE = 5
KLA_DTYPE_F32 = 0
KLA_DTYPE_BF16 = 1
KLA_BETA_KACZMARZ = 0
KLA_BETA_GIVEN = 1
_BETA_MODES = {"kaczmarz": KLA_BETA_KACZMARZ, "given": KLA_BETA_GIVEN}
CHUNK = 64

_lock = threading.Lock()
_lib = None


class KlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"KLA status {status}: {message}")
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_stale: bool = True) -> ctypes.CDLL:
    """Load libkla_gb300.so (compiling it first when sources are newer and
    nvcc is present).  Raises if the library is unavailable."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_stale and _build.is_stale():
            _build.build()
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError("libkla_gb300.so is missing; run __graft_entry__.build()")
        lib = ctypes.CDLL(_build.LIB_PATH)
        vp, fp, ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
        I, F, Z = ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.kla_status_str.restype = ctypes.c_char_p
        lib.kla_status_str.argtypes = [I]
        lib.kla_last_error_message.restype = ctypes.c_char_p
        lib.kla_last_error_message.argtypes = []
        lib.kla_version.restype = I
        lib.kla_version.argtypes = []
        lib.kla_launch_count.restype = ctypes.c_ulonglong
        lib.kla_launch_count.argtypes = []
        lib.kla_chunk_fwd_workspace_size.restype = Z
        lib.kla_chunk_fwd_workspace_size.argtypes = [I, I, I, I, I, I, I]
        lib.kla_chunk_fwd_varlen_workspace_size.restype = Z
        lib.kla_chunk_fwd_varlen_workspace_size.argtypes = [I, I, I, I, I, I, I]
        lib.kla_chunk_fwd.restype = I
        lib.kla_chunk_fwd.argtypes = [vp, vp, vp, fp, fp, F, fp, vp, fp,
                                      I, I, I, I, I, I, I, vp, Z, vp]
        lib.kla_chunk_fwd_varlen.restype = I
        lib.kla_chunk_fwd_varlen.argtypes = [vp, vp, vp, fp, fp, F, fp, vp, fp, ip,
                                             I, I, I, I, I, I, I, vp, Z, vp]
        lib.kla_decode_step.restype = I
        lib.kla_decode_step.argtypes = [vp, vp, vp, fp, fp, F, fp, vp, I, I, I, I, I, vp]
        lib.kla_chunk_fwd_ex.restype = I
        lib.kla_chunk_fwd_ex.argtypes = [vp, vp, vp, fp, fp, F, fp, vp, fp,
                                         I, I, I, I, I, I, I, I, vp, Z, vp]
        lib.kla_chunk_fwd_varlen_ex.restype = I
        lib.kla_chunk_fwd_varlen_ex.argtypes = [vp, vp, vp, fp, fp, F, fp, vp, fp, ip,
                                                I, I, I, I, I, I, I, I, vp, Z, vp]
        lib.kla_decode_step_ex.restype = I
        lib.kla_decode_step_ex.argtypes = [vp, vp, vp, fp, fp, F, fp, vp, I, I, I, I, I, I, vp]
        lib.kla_ccq_query_workspace_size.restype = Z
        lib.kla_ccq_query_workspace_size.argtypes = [I, I, I, I, I]
        lib.kla_ccq_query.restype = I
        lib.kla_ccq_query.argtypes = [vp, vp, fp, fp, fp, fp, vp, fp, fp, fp,
                                      I, I, I, I, I, vp, Z, vp]
        lib.kla_ccq_query_step.restype = I
        lib.kla_ccq_query_step.argtypes = [vp, vp, fp, fp, fp, fp, vp, I, I, I, I, vp]
        lib.kla_chunk_bwd_workspace_size.restype = Z
        lib.kla_chunk_bwd_workspace_size.argtypes = [I, I, I, I, I]
        lib.kla_chunk_bwd.restype = I
        lib.kla_chunk_bwd.argtypes = [vp, vp, vp, fp, fp, F, fp, vp, fp, vp, vp, vp, fp, fp, fp,
                                      I, I, I, I, I, I, I, I, vp, Z, vp]
        lib.kla_chunk_bwd_varlen_workspace_size.restype = Z
        lib.kla_chunk_bwd_varlen_workspace_size.argtypes = [I, I, I, I, I]
        lib.kla_chunk_bwd_varlen.restype = I
        lib.kla_chunk_bwd_varlen.argtypes = [vp, vp, vp, fp, fp, F, fp, vp, fp, vp, vp, vp, fp, fp,
                                             fp, ip, I, I, I, I, I, I, I, I, vp, Z, vp]
        lib.kla_chunk_fwd_noalloc.restype = I
        lib.kla_chunk_fwd_noalloc.argtypes = [vp, vp, vp, fp, fp, F, fp, vp, fp,
                                              I, I, I, I, I, I, I, vp]
        lib.kla_chunk_fwd_noalloc_status.restype = I
        lib.kla_chunk_fwd_noalloc_status.argtypes = [vp]
        lib.kla_workspace_status.restype = I
        lib.kla_workspace_status.argtypes = [vp, Z, vp]
        _lib = lib
        return lib


def _check(status: int):
    if status != KLA_OK:
        lib = load()
        raise KlaError(status, lib.kla_last_error_message().decode() or
                       lib.kla_status_str(status).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KLA_DTYPE_BF16
    if t.dtype == torch.float32:
        return KLA_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, name, dtype=None, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def kla_status_str(status: int) -> str:
    return load().kla_status_str(status).decode()


def kla_version() -> int:
    return load().kla_version()


def kla_launch_count() -> int:
    return int(load().kla_launch_count())


def kla_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk=CHUNK, dtype=KLA_DTYPE_BF16) -> int:
    return int(load().kla_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dtype))


def kla_chunk_fwd_varlen_workspace_size(N, total_T, H, dk, dv, chunk=CHUNK,
                                        dtype=KLA_DTYPE_BF16) -> int:
    return int(load().kla_chunk_fwd_varlen_workspace_size(N, total_T, H, dk, dv, chunk, dtype))


def _mode(beta_mode) -> int:
    if beta_mode not in _BETA_MODES:
        raise ValueError(f"beta_mode must be one of {sorted(_BETA_MODES)}")
    return _BETA_MODES[beta_mode]


def _workspace(nbytes, device, workspace):
    if nbytes == 0:
        # a path that needs none still records its status in a given workspace
        if workspace is None:
            return None, 0
        return workspace, workspace.numel() * workspace.element_size()
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    return workspace, workspace.numel() * workspace.element_size()


def kla_chunk_fwd(q, k, v, alpha, eta, eps, S0=None, o=None, S_T=None, workspace=None,
                  stream=None, chunk=CHUNK, return_final_state=True, beta_mode="kaczmarz"):
    """Chunkwise prefill; q,k: [B,T,H,dk], v: [B,T,H,dv], alpha,eta: [B,T,H]
    fp32 (alpha None: no decay), S0: [B,H,dk,dv] fp32 or None.  beta_mode
    "kaczmarz" (beta = eta / (||k||^2 + eps)) or "given" (beta = eta).
    Returns (o, S_T)."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _need(q, "q"); _need(k, "k", q.dtype, (B, T, H, dk)); _need(v, "v", q.dtype, (B, T, H, dv))
    _need(alpha, "alpha", torch.float32, (B, T, H)); _need(eta, "eta", torch.float32, (B, T, H))
    _need(S0, "S0", torch.float32, (B, H, dk, dv))
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    _need(o, "o", q.dtype, (B, T, H, dv))
    if S_T is None and return_final_state:
        S_T = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    _need(S_T, "S_T", torch.float32, (B, H, dk, dv))
    nbytes = int(lib.kla_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dt))
    workspace, wsb = _workspace(nbytes, q.device, workspace)
    st = lib.kla_chunk_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), float(eps),
                              _ptr(S0), _ptr(o), _ptr(S_T), B, T, H, dk, dv, chunk, dt,
                              _mode(beta_mode), _ptr(workspace), wsb, _stream(stream))
    _check(st)
    return o, S_T


def kla_chunk_bwd_workspace_size(B, T, H, dk, dtype=KLA_DTYPE_BF16) -> int:
    return int(load().kla_chunk_bwd_workspace_size(B, T, H, dk, dtype))


def kla_chunk_bwd(q, k, v, alpha, eta, eps, S0, d_o, dS_T=None, workspace=None, stream=None,
                  chunk=CHUNK, beta_mode="kaczmarz", want_dS0=True):
    """Backward of kla_chunk_fwd: the gradients of sum <d_o, o> + <dS_T, S_T>.
    Inputs as kla_chunk_fwd; d_o: [B,T,H,dv] in q's dtype; dS_T: [B,H,dk,dv]
    fp32 or None.  Returns (dq, dk, dv, dalpha, deta, dS0); dalpha is None when
    alpha is None, dS0 None unless want_dS0."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _need(q, "q"); _need(k, "k", q.dtype, (B, T, H, dk)); _need(v, "v", q.dtype, (B, T, H, dv))
    _need(alpha, "alpha", torch.float32, (B, T, H)); _need(eta, "eta", torch.float32, (B, T, H))
    _need(S0, "S0", torch.float32, (B, H, dk, dv)); _need(d_o, "d_o", q.dtype, (B, T, H, dv))
    _need(dS_T, "dS_T", torch.float32, (B, H, dk, dv))
    dq = torch.empty_like(q)
    dkk = torch.empty_like(k)
    dvv = torch.empty_like(v)
    dalpha = None if alpha is None else torch.empty_like(alpha)
    deta = torch.empty_like(eta)
    dS0 = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device) if want_dS0 else None
    nbytes = int(lib.kla_chunk_bwd_workspace_size(B, T, H, dk, dt))
    workspace, wsb = _workspace(nbytes, q.device, workspace)
    st = lib.kla_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), float(eps),
                           _ptr(S0), _ptr(d_o), _ptr(dS_T), _ptr(dq), _ptr(dkk), _ptr(dvv),
                           _ptr(dalpha), _ptr(deta), _ptr(dS0), B, T, H, dk, dv, chunk, dt,
                           _mode(beta_mode), _ptr(workspace), wsb, _stream(stream))
    _check(st)
    return dq, dkk, dvv, dalpha, deta, dS0


def kla_chunk_bwd_varlen_workspace_size(N, total_T, H, dk, dtype=KLA_DTYPE_BF16) -> int:
    return int(load().kla_chunk_bwd_varlen_workspace_size(N, total_T, H, dk, dtype))


def kla_chunk_bwd_varlen(q, k, v, alpha, eta, eps, cu_seqlens, S0, d_o, dS_T=None,
                         workspace=None, stream=None, chunk=CHUNK, beta_mode="kaczmarz",
                         want_dS0=True):
    """Backward of kla_chunk_fwd_varlen: packed q, k: [total_T,H,dk], v, d_o:
    [total_T,H,dv], alpha, eta: [total_T,H] fp32, cu_seqlens: int32 [N+1] on the
    device, S0, dS_T: [N,H,dk,dv] fp32 or None.  Returns (dq, dk, dv, dalpha,
    deta, dS0) like kla_chunk_bwd."""
    lib = load()
    total_T, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.shape[0] - 1
    dt = _dtype_code(q)
    _need(q, "q"); _need(k, "k", q.dtype, (total_T, H, dk)); _need(v, "v", q.dtype, (total_T, H, dv))
    _need(alpha, "alpha", torch.float32, (total_T, H)); _need(eta, "eta", torch.float32, (total_T, H))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (N + 1,))
    _need(S0, "S0", torch.float32, (N, H, dk, dv)); _need(d_o, "d_o", q.dtype, (total_T, H, dv))
    _need(dS_T, "dS_T", torch.float32, (N, H, dk, dv))
    dq, dkk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dalpha = None if alpha is None else torch.empty_like(alpha)
    deta = torch.empty_like(eta)
    dS0 = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device) if want_dS0 else None
    nbytes = int(lib.kla_chunk_bwd_varlen_workspace_size(N, total_T, H, dk, dt))
    workspace, wsb = _workspace(nbytes, q.device, workspace)
    st = lib.kla_chunk_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), float(eps),
                                  _ptr(S0), _ptr(d_o), _ptr(dS_T), _ptr(dq), _ptr(dkk), _ptr(dvv),
                                  _ptr(dalpha), _ptr(deta), _ptr(dS0), _ptr(cu_seqlens), N,
                                  total_T, H, dk, dv, chunk, dt, _mode(beta_mode),
                                  _ptr(workspace), wsb, _stream(stream))
    _check(st)
    return dq, dkk, dvv, dalpha, deta, dS0


class _KlaChunk(torch.autograd.Function):
    """kla_chunk_fwd as an autograd function: its backward is kla_chunk_bwd."""

    @staticmethod
    def forward(ctx, q, k, v, alpha, eta, S0, eps, beta_mode):
        o, S_T = kla_chunk_fwd(q, k, v, alpha, eta, eps, S0, beta_mode=beta_mode)
        ctx.save_for_backward(q, k, v, alpha, eta, S0)
        ctx.has_alpha, ctx.has_S0 = alpha is not None, S0 is not None
        ctx.eps, ctx.beta_mode = eps, beta_mode
        return o, S_T

    @staticmethod
    def backward(ctx, d_o, dS_T):
        q, k, v, alpha, eta, S0 = ctx.saved_tensors
        alpha = alpha if ctx.has_alpha else None
        S0 = S0 if ctx.has_S0 else None
        if d_o is None:
            d_o = torch.zeros_like(v)
        dq, dk, dv, da, de, dS0 = kla_chunk_bwd(
            q, k, v, alpha, eta, ctx.eps, S0, d_o.contiguous().to(q.dtype),
            None if dS_T is None else dS_T.contiguous().float(), beta_mode=ctx.beta_mode,
            want_dS0=ctx.has_S0)
        return dq, dk, dv, da, de, dS0, None, None


def kla_chunk(q, k, v, alpha, eta, eps, S0=None, beta_mode="kaczmarz"):
    """Differentiable chunkwise forward: (o, S_T) = kla_chunk_fwd(...), with
    gradients for q, k, v, alpha, eta and S0 from kla_chunk_bwd."""
    return _KlaChunk.apply(q, k, v, alpha, eta, S0, float(eps), beta_mode)


def kla_chunk_fwd_noalloc(q, k, v, alpha, eta, eps, S0=None, o=None, S_T=None, stream=None,
                          chunk=CHUNK):
    """kla_chunk_fwd for callers that cannot allocate device memory while the
    prefill runs: the library uses its built-in device array as workspace
    (sizes that need more than KLA_NOALLOC_SCRATCH_BYTES raise KlaError).
    Calls sharing that array must not overlap on the GPU.  Pass ``o`` and
    ``S_T`` to avoid any allocation here as well.  Returns (o, S_T)."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _need(q, "q"); _need(k, "k", q.dtype, (B, T, H, dk)); _need(v, "v", q.dtype, (B, T, H, dv))
    _need(alpha, "alpha", torch.float32, (B, T, H)); _need(eta, "eta", torch.float32, (B, T, H))
    _need(S0, "S0", torch.float32, (B, H, dk, dv))
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    _need(o, "o", q.dtype, (B, T, H, dv))
    _need(S_T, "S_T", torch.float32, (B, H, dk, dv))
    st = lib.kla_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), float(eps),
                                   _ptr(S0), _ptr(o), _ptr(S_T), B, T, H, dk, dv, chunk, dt,
                                   _stream(stream))
    _check(st)
    return o, S_T


def kla_chunk_fwd_noalloc_status(stream=None) -> int:
    """Synchronises the stream and returns the device status that the last
    kla_chunk_fwd_noalloc call on the current device recorded in the built-in
    array (raises KlaError when it is not OK)."""
    st = load().kla_chunk_fwd_noalloc_status(_stream(stream))
    _check(st)
    return st


def kla_chunk_fwd_varlen(q, k, v, alpha, eta, eps, cu_seqlens, S0=None, o=None, S_T=None,
                         workspace=None, stream=None, chunk=CHUNK, return_final_state=True,
                         check_status=False, beta_mode="kaczmarz"):
    """Packed prefill; q,k: [total_T,H,dk], v: [total_T,H,dv], alpha,eta:
    [total_T,H], cu_seqlens: int32 [N+1] on the device.  Returns (o, S_T)."""
    lib = load()
    total, H, dk = q.shape
    dv = v.shape[-1]
    N = cu_seqlens.shape[0] - 1
    dt = _dtype_code(q)
    _need(q, "q"); _need(k, "k", q.dtype, (total, H, dk)); _need(v, "v", q.dtype, (total, H, dv))
    _need(alpha, "alpha", torch.float32, (total, H)); _need(eta, "eta", torch.float32, (total, H))
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    _need(S0, "S0", torch.float32, (N, H, dk, dv))
    if o is None:
        o = torch.empty((total, H, dv), dtype=q.dtype, device=q.device)
    _need(o, "o", q.dtype, (total, H, dv))
    if S_T is None and return_final_state:
        S_T = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    _need(S_T, "S_T", torch.float32, (N, H, dk, dv))
    nbytes = int(lib.kla_chunk_fwd_varlen_workspace_size(N, total, H, dk, dv, chunk, dt))
    workspace, wsb = _workspace(nbytes, q.device, workspace)
    s = _stream(stream)
    st = lib.kla_chunk_fwd_varlen_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta),
                                     float(eps), _ptr(S0), _ptr(o), _ptr(S_T), _ptr(cu_seqlens),
                                     N, total, H, dk, dv, chunk, dt, _mode(beta_mode),
                                     _ptr(workspace), wsb, s)
    _check(st)
    if check_status:
        _check(lib.kla_workspace_status(_ptr(workspace), wsb, s))
    return o, S_T


def kla_decode_step(q, k, v, alpha, eta, eps, S, o=None, stream=None, beta_mode="kaczmarz"):
    """One decode step; q,k: [B,H,dk], v: [B,H,dv], alpha,eta: [B,H], S:
    [B,H,dk,dv] fp32 updated in place.  Returns o [B,H,dv]."""
    lib = load()
    B, H, dk = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    _need(q, "q"); _need(k, "k", q.dtype, (B, H, dk)); _need(v, "v", q.dtype, (B, H, dv))
    _need(alpha, "alpha", torch.float32, (B, H)); _need(eta, "eta", torch.float32, (B, H))
    _need(S, "S", torch.float32, (B, H, dk, dv))
    if o is None:
        o = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    _need(o, "o", q.dtype, (B, H, dv))
    st = lib.kla_decode_step_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), float(eps),
                                _ptr(S), _ptr(o), B, H, dk, dv, dt, _mode(beta_mode),
                                _stream(stream))
    _check(st)
    return o


def kla_workspace_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns the device status recorded in
    ``workspace`` (raises KlaError when it is not OK)."""
    lib = load()
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.kla_workspace_status(_ptr(workspace), wsb, _stream(stream))
    _check(st)
    return st


# The *_ex C entry points: the same calls with the write-coefficient mode as a
# required argument ("kaczmarz" or "given").
def kla_chunk_fwd_ex(q, k, v, alpha, eta, eps, beta_mode, S0=None, **kw):
    return kla_chunk_fwd(q, k, v, alpha, eta, eps, S0, beta_mode=beta_mode, **kw)


def kla_chunk_fwd_varlen_ex(q, k, v, alpha, eta, eps, cu_seqlens, beta_mode, S0=None, **kw):
    return kla_chunk_fwd_varlen(q, k, v, alpha, eta, eps, cu_seqlens, S0, beta_mode=beta_mode,
                                **kw)


def kla_decode_step_ex(q, k, v, alpha, eta, eps, S, beta_mode, **kw):
    return kla_decode_step(q, k, v, alpha, eta, eps, S, beta_mode=beta_mode, **kw)



def kla_ccq_query_workspace_size(B, T, H, dk, dtype=KLA_DTYPE_BF16) -> int:
    return int(load().kla_ccq_query_workspace_size(B, T, H, dk, dtype))


def kla_ccq_query(q, k, lam, stats0=None, q_clean=None, return_stats=True, workspace=None,
                  stream=None):
    """Curvature-Conditioned Query contraction: q_clean = (I - lam Sigma_t) q with
    Sigma_t the running covariance of the keys.  q, k: [B,T,H,dk]; lam: [B,T,H]
    fp32; stats0: None or (Ms [B,H,dk,dk], ms [B,H,dk], ns [B,H]) fp32.
    Returns (q_clean, stats_T); a CCQ layer is kla_chunk_fwd(q_clean, k, ...)."""
    lib = load()
    B, T, H, dk = q.shape
    dt = _dtype_code(q)
    _need(q, "q"); _need(k, "k", q.dtype, (B, T, H, dk)); _need(lam, "lam", torch.float32, (B, T, H))
    M0 = m0 = n0 = None
    if stats0 is not None:
        M0, m0, n0 = stats0
        _need(M0, "Ms0", torch.float32, (B, H, dk, dk)); _need(m0, "ms0", torch.float32, (B, H, dk))
        _need(n0, "ns0", torch.float32, (B, H))
    if q_clean is None:
        q_clean = torch.empty_like(q)
    _need(q_clean, "q_clean", q.dtype, (B, T, H, dk))
    Ms = ms = ns = None
    if return_stats:
        Ms = torch.empty((B, H, dk, dk), dtype=torch.float32, device=q.device)
        ms = torch.empty((B, H, dk), dtype=torch.float32, device=q.device)
        ns = torch.empty((B, H), dtype=torch.float32, device=q.device)
    nbytes = int(lib.kla_ccq_query_workspace_size(B, T, H, dk, dt))
    workspace, wsb = _workspace(nbytes, q.device, workspace)
    st = lib.kla_ccq_query(_ptr(q), _ptr(k), _ptr(lam), _ptr(M0), _ptr(m0), _ptr(n0),
                           _ptr(q_clean), _ptr(Ms), _ptr(ms), _ptr(ns), B, T, H, dk, dt,
                           _ptr(workspace), wsb, _stream(stream))
    _check(st)
    return q_clean, (Ms, ms, ns)


def kla_ccq_query_step(q, k, lam, Ms, ms, ns, q_clean=None, stream=None):
    """One CCQ token per (b, h): the statistics (Ms, ms, ns) are updated in place
    with k; returns q_clean [B,H,dk]."""
    lib = load()
    B, H, dk = q.shape
    dt = _dtype_code(q)
    _need(q, "q"); _need(k, "k", q.dtype, (B, H, dk)); _need(lam, "lam", torch.float32, (B, H))
    _need(Ms, "Ms", torch.float32, (B, H, dk, dk)); _need(ms, "ms", torch.float32, (B, H, dk))
    _need(ns, "ns", torch.float32, (B, H))
    if q_clean is None:
        q_clean = torch.empty_like(q)
    _need(q_clean, "q_clean", q.dtype, (B, H, dk))
    st = lib.kla_ccq_query_step(_ptr(q), _ptr(k), _ptr(lam), _ptr(Ms), _ptr(ms), _ptr(ns),
                                _ptr(q_clean), B, H, dk, dt, _stream(stream))
    _check(st)
    return q_clean
