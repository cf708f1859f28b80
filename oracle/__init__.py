"""fp64 CPU oracle for Kaczmarz Linear Attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or executes anything here, and this
package imports nothing from the product.

The arithmetic lives in ``kla_oracle.c`` (plain sequential fp64 recurrence,
see the header there for the passages it follows).  This module only
compiles it with gcc, converts arrays to contiguous float64 and calls it.

Functions
---------
forward(q, k, v, alpha, eta, eps, S0=None, nthreads=1) -> (o, S_T)
    fixed-length batch, q,k: [B,T,H,dk], v: [B,T,H,dv], alpha,eta: [B,T,H],
    S0: [B,H,dk,dv] or None.
forward_varlen(q, k, v, alpha, eta, eps, cu_seqlens, S0=None, nthreads=1)
    packed batch, q,k: [total_T,H,dk], cu_seqlens: [N+1] int.
backward(q, k, v, alpha, eta, eps, S0, do, dS_T=None, nthreads=1)
    -> (dq, dk, dv, dalpha, deta, dS0): the gradient of
    L = sum <do, o> + <dS_T, S_T> by reverse-mode differentiation of the
    recurrence (``kla_oracle_bwd.c``); dalpha is None when alpha is None.
decode(q, k, v, alpha, eta, eps, S, nthreads=1) -> (o, S_new)
    one token per (b,h): q,k: [B,H,dk], v: [B,H,dv], alpha,eta: [B,H],
    S: [B,H,dk,dv].  The decode step is the same recurrence applied to a
    single token on a stored state, so it calls ``forward`` with T = 1.

Every array argument may be a numpy array or a CPU torch tensor of any
floating dtype; values are upcast exactly to float64 (bf16 and fp32 are
subsets of fp64).

Every function also takes ``beta_mode``: "kaczmarz" (default, beta_t =
eta_t / (||k_t||^2 + eps)) or "given" (beta_t = eta_t, the learned write
strength of Gated DeltaNet); and ``alpha`` may be None (alpha_t = 1, no
decay: DeltaNet).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kla_oracle.c")
_SRC_CCQ = os.path.join(_HERE, "ccq_oracle.c")
_SRC_BWD = os.path.join(_HERE, "kla_oracle_bwd.c")
_LIB_PATH = os.path.join(_HERE, "libkla_oracle.so")
_lock = threading.Lock()
_lib = None


def _elf_matches_host(path: str) -> bool:
    import platform
    want = {"x86_64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine())
    with open(path, "rb") as f:
        head = f.read(20)
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return False
    return want is None or int.from_bytes(head[18:20], "little") == want


def build(force: bool = False) -> str:
    """Compile kla_oracle.c into libkla_oracle.so next to it (gcc, -O2, no
    fast-math, no host-specific flags so it builds the same on x86 and Arm)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                                  os.path.getmtime(_SRC_CCQ),
                                                  os.path.getmtime(_SRC_BWD))
             or not _elf_matches_host(_LIB_PATH))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, _SRC_CCQ, _SRC_BWD]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int)
    lib.kla_oracle_forward.restype = ctypes.c_int
    lib.kla_oracle_forward.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        dp, dp, dp, dp, dp, ctypes.c_double, dp, dp, dp, ctypes.c_int]
    lib.kla_oracle_forward_varlen.restype = ctypes.c_int
    lib.kla_oracle_forward_varlen.argtypes = [
        ctypes.c_int, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        dp, dp, dp, dp, dp, ctypes.c_double, dp, dp, dp, ctypes.c_int]
    lib.kla_oracle_forward_ex.restype = ctypes.c_int
    lib.kla_oracle_forward_ex.argtypes = lib.kla_oracle_forward.argtypes + [ctypes.c_int]
    lib.kla_oracle_forward_varlen_ex.restype = ctypes.c_int
    lib.kla_oracle_forward_varlen_ex.argtypes = lib.kla_oracle_forward_varlen.argtypes + [ctypes.c_int]
    if hasattr(lib, "kla_oracle_backward"):
        lib.kla_oracle_backward.restype = ctypes.c_int
        lib.kla_oracle_backward.argtypes = (
            [ctypes.c_int] * 5 + [dp] * 5 + [ctypes.c_double] + [dp] * 9 + [ctypes.c_int] * 2)
    if hasattr(lib, "ccq_oracle_query"):
        lib.ccq_oracle_query.restype = ctypes.c_int
        lib.ccq_oracle_query.argtypes = [ctypes.c_int] * 4 + [dp] * 10
    return lib


_MODES = {"kaczmarz": 0, "given": 1}


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def compile_variant(source_text: str, so_path: str):
    """Compiles a modified copy of the oracle source (used by the tests that
    plant mistakes in the oracle to show the pins catch them) and returns an
    object with the same ``forward`` function as this module."""
    src_path = so_path[:-3] + ".c"
    with open(src_path, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                    "-ffp-contract=off", "-o", so_path, src_path], check=True)
    lib = _bind(ctypes.CDLL(so_path))

    class _Variant:
        @staticmethod
        def forward(q, k, v, alpha, eta, eps, S0=None, nthreads=1, beta_mode="kaczmarz"):
            return _forward_with(lib, q, k, v, alpha, eta, eps, S0, nthreads, beta_mode)
    return _Variant


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor (CPU); exact upcast
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def forward(q, k, v, alpha, eta, eps, S0=None, nthreads: int = 1, beta_mode: str = "kaczmarz"):
    return _forward_with(_load(), q, k, v, alpha, eta, eps, S0, nthreads, beta_mode)


def _forward_with(lib, q, k, v, alpha, eta, eps, S0, nthreads, beta_mode="kaczmarz"):
    q, k, v, alpha, eta, S0 = map(_f64, (q, k, v, alpha, eta, S0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (B, T, H, dk) and v.shape == (B, T, H, dv)
    assert (alpha is None or alpha.shape == (B, T, H)) and eta.shape == (B, T, H)
    if S0 is not None:
        assert S0.shape == (B, H, dk, dv)
    o = np.zeros((B, T, H, dv), dtype=np.float64)
    S = np.zeros((B, H, dk, dv), dtype=np.float64)
    rc = lib.kla_oracle_forward_ex(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(alpha), _ptr(eta), float(eps), _ptr(S0),
                                   _ptr(o), _ptr(S), int(nthreads), _MODES[beta_mode])
    if rc != 0:
        raise RuntimeError(f"kla_oracle_forward failed rc={rc}")
    return o, S


def forward_varlen(q, k, v, alpha, eta, eps, cu_seqlens, S0=None, nthreads: int = 1,
                   beta_mode: str = "kaczmarz"):
    lib = _load()
    q, k, v, alpha, eta, S0 = map(_f64, (q, k, v, alpha, eta, S0))
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
        dtype=np.int32))
    N = cu.shape[0] - 1
    total, H, dk = q.shape
    dv = v.shape[-1]
    assert int(cu[-1]) == total
    if S0 is not None:
        assert S0.shape == (N, H, dk, dv)
    o = np.zeros((total, H, dv), dtype=np.float64)
    S = np.zeros((N, H, dk, dv), dtype=np.float64)
    rc = lib.kla_oracle_forward_varlen_ex(
        N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), H, dk, dv,
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), float(eps), _ptr(S0),
        _ptr(o), _ptr(S), int(nthreads), _MODES[beta_mode])
    if rc != 0:
        raise RuntimeError(f"kla_oracle_forward_varlen failed rc={rc}")
    return o, S


def decode(q, k, v, alpha, eta, eps, S, nthreads: int = 1, beta_mode: str = "kaczmarz"):
    q, k, v, alpha, eta, S = map(_f64, (q, k, v, alpha, eta, S))
    B, H, dk = q.shape
    o, S_new = forward(q[:, None], k[:, None], v[:, None],
                       None if alpha is None else alpha[:, None],
                       eta[:, None], eps, S, nthreads=nthreads, beta_mode=beta_mode)
    return o[:, 0], S_new


def ccq_query(q, k, lam, stats0=None):
    """CCQ read-side contraction (see ccq_oracle.c): q_clean_t = (I - lambda_t
    Sigma_t) q_t with Sigma_t the running population covariance of the keys up
    to token t.  q, k: [B,T,H,dk]; lam: [B,T,H]; stats0: None or (Ms [B,H,dk,dk],
    ms [B,H,dk], ns [B,H]).  Returns (q_clean, (Ms, ms, ns)).  The CCQ layer
    output is ``forward(q_clean, k, v, ...)``: the write rule is unchanged."""
    lib = _load()
    q, k, lam = map(_f64, (q, k, lam))
    B, T, H, dk = q.shape
    assert k.shape == q.shape and lam.shape == (B, T, H)
    M0 = m0 = n0 = None
    if stats0 is not None:
        M0, m0, n0 = map(_f64, stats0)
    qc = np.zeros_like(q)
    Ms = np.zeros((B, H, dk, dk)); ms = np.zeros((B, H, dk)); ns = np.zeros((B, H))
    rc = lib.ccq_oracle_query(B, T, H, dk, _ptr(q), _ptr(k), _ptr(lam), _ptr(M0), _ptr(m0),
                              _ptr(n0), _ptr(qc), _ptr(Ms), _ptr(ms), _ptr(ns))
    if rc != 0:
        raise RuntimeError(f"ccq_oracle_query failed rc={rc}")
    return qc, (Ms, ms, ns)


def backward(q, k, v, alpha, eta, eps, S0, do, dS_T=None, nthreads: int = 1,
             beta_mode: str = "kaczmarz"):
    """Gradient of L = sum_t <do_t, o_t> + <dS_T, S_T> for the fixed-length
    forward (see kla_oracle_bwd.c).  Returns (dq, dk, dv, dalpha, deta, dS0)."""
    return _backward_with(_load(), q, k, v, alpha, eta, eps, S0, do, dS_T, nthreads, beta_mode)


def _backward_with(lib, q, k, v, alpha, eta, eps, S0, do, dS_T, nthreads, beta_mode):
    q, k, v, alpha, eta, S0, do, dS_T = map(_f64, (q, k, v, alpha, eta, S0, do, dS_T))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (B, T, H, dk) and v.shape == (B, T, H, dv) and do.shape == v.shape
    assert (alpha is None or alpha.shape == (B, T, H)) and eta.shape == (B, T, H)
    for x in (S0, dS_T):
        assert x is None or x.shape == (B, H, dk, dv)
    dq = np.zeros_like(q); dkk = np.zeros_like(k); dvv = np.zeros_like(v)
    da = None if alpha is None else np.zeros_like(alpha)
    de = np.zeros_like(eta)
    dS0 = np.zeros((B, H, dk, dv))
    rc = lib.kla_oracle_backward(B, T, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                 _ptr(eta), float(eps), _ptr(S0), _ptr(do), _ptr(dS_T),
                                 _ptr(dq), _ptr(dkk), _ptr(dvv), _ptr(da), _ptr(de),
                                 _ptr(dS0), int(nthreads), _MODES[beta_mode])
    if rc != 0:
        raise RuntimeError(f"kla_oracle_backward failed rc={rc}")
    return dq, dkk, dvv, da, de, dS0


def source_bwd() -> str:
    with open(_SRC_BWD) as f:
        return f.read()


def compile_bwd_variant(source_text: str, so_path: str):
    """Compiles a modified copy of kla_oracle_bwd.c (for the tests that plant
    mistakes in it) and returns an object with the same ``backward``."""
    src_path = so_path[:-3] + ".c"
    with open(src_path, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                    "-ffp-contract=off", "-o", so_path, src_path], check=True)
    lib = ctypes.CDLL(so_path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.kla_oracle_backward.restype = ctypes.c_int
    lib.kla_oracle_backward.argtypes = (
        [ctypes.c_int] * 5 + [dp] * 5 + [ctypes.c_double] + [dp] * 9 + [ctypes.c_int] * 2)

    class _Variant:
        @staticmethod
        def backward(q, k, v, alpha, eta, eps, S0, do, dS_T=None, nthreads=1,
                     beta_mode="kaczmarz"):
            return _backward_with(lib, q, k, v, alpha, eta, eps, S0, do, dS_T, nthreads,
                                  beta_mode)
    return _Variant
