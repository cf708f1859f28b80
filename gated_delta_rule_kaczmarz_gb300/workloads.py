"""Seeded synthetic inputs for Kaczmarz Linear Attention workloads.

This module draws random numbers and rounds them to the storage dtype; it
holds none of the method's arithmetic.  Both the CUDA path (tests, bench) and
the fp64 oracle consume exactly the tensors it returns.

Distributions (the conventions used throughout):
  * N(0, x) has variance x; lognormal(0, s) is exp(N(0, s^2)) (s is the
    standard deviation of the log).
  * q ~ N(0, 1/dk); k = N(0, 1/dk) * f with one norm factor f ~ lognormal per
    (token, head) row; v ~ N(0, 1).
  * alpha = exp(-softplus(x)) = sigmoid(-x), x ~ N(0,1): a scalar decay per
    token and head in (0, 1).
  * eta = sigmoid(x), x ~ N(0,1), or eta = 1 where a workload fixes it.
  * S0 ~ N(0, s0_var) in fp32, or absent (zero state).
Generator: numpy PCG64(seed); arrays are drawn in the fixed order
q, k, norm factor, v, alpha noise, eta noise, S0 (decode draws S first).
q, k, v are rounded to bf16 (round-to-nearest-even) where the workload is bf16;
alpha, eta and the states are always fp32.

Named workloads (sizes of the Kaczmarz Linear Attention setting: a 0.4B-scale
layer, a 32K-token context, batched decode and packed variable-length
prefill):
  tiny_fp32     B=1 H=2 T=256 d=64 fp32, S0=0, norm lognormal(0,0.5), seed 0
  layer_prefill B=4 H=8 T=2048 d=128 bf16, S0~N(0,0.01), seed 1
  long_context  B=1 H=16 T=32768 d=128 bf16, norm lognormal(0,1), eta=1,
                S0=0, seed 2
  decode_b256   B=256 H=16 d=128, 64 single-token steps, S~N(0,0.01), seed 3
  varlen_64     64 sequences, lengths uniform in [128, 8192], H=16 d=128
                bf16, S0~N(0,0.01) per sequence, seed 4
All use eps = 1e-6 and chunk length 64.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

EPS_DEFAULT = 1e-6
CHUNK = 64


def _dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def _normal(rng, shape, std):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def _decay(rng, shape):
    x = rng.standard_normal(size=shape)  # float64
    # exp(-softplus(x)) written as a logistic of -x
    return (1.0 / (1.0 + np.exp(x))).astype(np.float32)


def _gate(rng, shape):
    x = rng.standard_normal(size=shape)
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


def _to(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(_dtype(dtype))


def _keys(rng, shape, dk, norm_sigma):
    k = _normal(rng, shape, 1.0 / np.sqrt(dk))
    f = np.exp(_normal(rng, shape[:-1], norm_sigma)).astype(np.float32)
    k *= f[..., None]
    return k


def prefill_inputs(B, T, H, dk, dv, dtype="bf16", seed=0, key_norm_sigma=0.5,
                   eta_one=False, s0_var=0.0, eps=EPS_DEFAULT):
    """Fixed-length batch: q,k [B,T,H,dk], v [B,T,H,dv], alpha,eta [B,T,H],
    S0 [B,H,dk,dv] (None when s0_var == 0)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal(rng, (B, T, H, dk), 1.0 / np.sqrt(dk))
    k = _keys(rng, (B, T, H, dk), dk, key_norm_sigma)
    v = _normal(rng, (B, T, H, dv), 1.0)
    alpha = _decay(rng, (B, T, H))
    eta = np.ones((B, T, H), np.float32) if eta_one else _gate(rng, (B, T, H))
    S0 = None
    if s0_var > 0:
        S0 = torch.from_numpy(_normal(rng, (B, H, dk, dv), float(np.sqrt(s0_var))))
    return dict(q=_to(q, dtype), k=_to(k, dtype), v=_to(v, dtype),
                alpha=torch.from_numpy(alpha), eta=torch.from_numpy(eta),
                S0=S0, eps=float(eps))


def varlen_lengths(N, lo, hi, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(lo, hi + 1, size=N).astype(np.int64)


def varlen_inputs(lengths, H, dk, dv, dtype="bf16", seed=0, key_norm_sigma=0.5,
                  eta_one=False, s0_var=0.0, eps=EPS_DEFAULT):
    """Packed batch: q,k [total_T,H,dk], v [total_T,H,dv], alpha,eta
    [total_T,H], cu_seqlens int32 [N+1], S0 [N,H,dk,dv] or None."""
    lengths = np.asarray(lengths, dtype=np.int64)
    N = int(lengths.shape[0])
    cu = np.zeros(N + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    total = int(cu[-1])
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    q = _normal(rng, (total, H, dk), 1.0 / np.sqrt(dk))
    k = _keys(rng, (total, H, dk), dk, key_norm_sigma)
    v = _normal(rng, (total, H, dv), 1.0)
    alpha = _decay(rng, (total, H))
    eta = np.ones((total, H), np.float32) if eta_one else _gate(rng, (total, H))
    S0 = None
    if s0_var > 0:
        S0 = torch.from_numpy(_normal(rng, (N, H, dk, dv), float(np.sqrt(s0_var))))
    return dict(q=_to(q, dtype), k=_to(k, dtype), v=_to(v, dtype),
                alpha=torch.from_numpy(alpha), eta=torch.from_numpy(eta),
                S0=S0, cu_seqlens=torch.from_numpy(cu), eps=float(eps))


def decode_inputs(B, H, dk, dv, steps, dtype="bf16", seed=0, key_norm_sigma=0.5,
                  s0_var=0.01, eps=EPS_DEFAULT):
    """Batched single-token decode: S [B,H,dk,dv] fp32, then per step
    q,k [steps,B,H,dk], v [steps,B,H,dv], alpha,eta [steps,B,H]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    S = _normal(rng, (B, H, dk, dv), float(np.sqrt(s0_var)))
    q = _normal(rng, (steps, B, H, dk), 1.0 / np.sqrt(dk))
    k = _keys(rng, (steps, B, H, dk), dk, key_norm_sigma)
    v = _normal(rng, (steps, B, H, dv), 1.0)
    alpha = _decay(rng, (steps, B, H))
    eta = _gate(rng, (steps, B, H))
    return dict(S=torch.from_numpy(S), q=_to(q, dtype), k=_to(k, dtype),
                v=_to(v, dtype), alpha=torch.from_numpy(alpha),
                eta=torch.from_numpy(eta), eps=float(eps))


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                      # "prefill" | "decode" | "varlen"
    dtype: str
    H: int
    d: int
    B: int = 1
    T: int = 0
    steps: int = 0
    N: int = 0
    len_lo: int = 0
    len_hi: int = 0
    key_norm_sigma: float = 0.5
    eta_one: bool = False
    s0_var: float = 0.0
    seed: int = 0
    chunk: int = CHUNK
    eps: float = EPS_DEFAULT
    extra: dict = field(default_factory=dict)

    def make(self, **overrides):
        """Draw this workload's inputs; ``overrides`` may shrink sizes
        (B, T, H, steps, N, len_lo, len_hi) for quick parity cases."""
        p = {f: getattr(self, f) for f in ("B", "T", "H", "d", "steps", "N",
                                           "len_lo", "len_hi", "seed")}
        p.update(overrides)
        if self.kind == "prefill":
            return prefill_inputs(p["B"], p["T"], p["H"], p["d"], p["d"], self.dtype,
                                  p["seed"], self.key_norm_sigma, self.eta_one,
                                  self.s0_var, self.eps)
        if self.kind == "decode":
            return decode_inputs(p["B"], p["H"], p["d"], p["d"], p["steps"], self.dtype,
                                 p["seed"], self.key_norm_sigma, self.s0_var, self.eps)
        if self.kind == "varlen":
            lens = varlen_lengths(p["N"], p["len_lo"], p["len_hi"], p["seed"])
            return varlen_inputs(lens, p["H"], p["d"], p["d"], self.dtype, p["seed"],
                                 self.key_norm_sigma, self.eta_one, self.s0_var,
                                 self.eps)
        raise ValueError(self.kind)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", "prefill", "fp32", H=2, d=64, B=1, T=256,
                          key_norm_sigma=0.5, s0_var=0.0, seed=0),
    "layer_prefill": Workload("layer_prefill", "prefill", "bf16", H=8, d=128, B=4,
                              T=2048, key_norm_sigma=0.5, s0_var=0.01, seed=1),
    "long_context": Workload("long_context", "prefill", "bf16", H=16, d=128, B=1,
                             T=32768, key_norm_sigma=1.0, eta_one=True,
                             s0_var=0.0, seed=2),
    "decode_b256": Workload("decode_b256", "decode", "bf16", H=16, d=128, B=256,
                            steps=64, key_norm_sigma=0.5, s0_var=0.01, seed=3),
    "varlen_64": Workload("varlen_64", "varlen", "bf16", H=16, d=128, N=64,
                          len_lo=128, len_hi=8192, key_norm_sigma=0.5,
                          s0_var=0.01, seed=4),
}
