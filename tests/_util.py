"""Shared test helpers: error measure and tolerances.

Tolerance (max abs error / max |reference|, per output tensor): 1e-4 for
fp32 inputs, 2e-2 for bf16 inputs with fp32 state.
"""
import numpy as np
import torch

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def rel_err(got, ref) -> float:
    got = got.detach().to("cpu", torch.float64).numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    scale = np.abs(ref).max()
    if scale == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / scale)


def cuda(d, keys=None):
    out = {}
    for name, x in d.items():
        if isinstance(x, torch.Tensor) and (keys is None or name in keys):
            out[name] = x.cuda()
        else:
            out[name] = x
    return out
