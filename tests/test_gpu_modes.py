"""GPU parity of the write-coefficient modes against the fp64 oracle: the
Kaczmarz coefficient and a given beta (Gated DeltaNet), each with and
without decay (alpha = None: DeltaNet), on every path (fp32 and bf16
prefill, varlen, decode).  Error measure and bounds as in the other parity
tests: max|gpu - oracle| / max|oracle|, 1e-4 (fp32) and 2e-2 (bf16)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300.workloads import decode_inputs, prefill_inputs, varlen_inputs
from tests._util import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu

MODES = [("kaczmarz", True), ("given", True), ("kaczmarz", False), ("given", False)]


def _given_eta(inp):
    # a learned beta in (0, 1/2): scaled eta, typical of a sigmoid gate
    return inp["eta"] * 0.5


@pytest.mark.parametrize("mode,decay", MODES)
@pytest.mark.parametrize("B,T,H,d,dtype", [(2, 200, 2, 64, "fp32"), (2, 257, 2, 128, "bf16"),
                                           (2, 256, 2, 128, "bf16")])
def test_prefill_modes(mode, decay, B, T, H, d, dtype):
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=70 + T, s0_var=0.01)
    if mode == "given":
        inp["eta"] = _given_eta(inp)
    if not decay:
        inp["alpha"] = None
    dv = cuda(inp)
    o, S = kla.kla_chunk_fwd(dv["q"], dv["k"], dv["v"], dv["alpha"], dv["eta"], dv["eps"],
                             dv["S0"], beta_mode=mode)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                  inp["eps"], inp["S0"], nthreads=8, beta_mode=mode)
    tol = TOL[inp["q"].dtype]
    assert rel_err(o, o_ref) <= tol
    assert rel_err(S, S_ref) <= tol


@pytest.mark.parametrize("mode,decay", MODES)
def test_varlen_modes(mode, decay):
    lens = [1, 63, 64, 130, 0, 200]
    inp = varlen_inputs(lens, 2, 128, 128, "bf16", seed=80, s0_var=0.01)
    if mode == "given":
        inp["eta"] = _given_eta(inp)
    if not decay:
        inp["alpha"] = None
    d = cuda(inp)
    o, S = kla.kla_chunk_fwd_varlen(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"],
                                    d["cu_seqlens"], d["S0"], check_status=True, beta_mode=mode)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_varlen(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                         inp["eps"], inp["cu_seqlens"], inp["S0"], nthreads=8,
                                         beta_mode=mode)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2


@pytest.mark.parametrize("mode,decay", MODES)
@pytest.mark.parametrize("d,dtype", [(64, "fp32"), (128, "bf16")])
def test_decode_modes(mode, decay, d, dtype):
    inp = decode_inputs(3, 4, d, d, steps=5, dtype=dtype, seed=90 + d)
    if mode == "given":
        inp["eta"] = inp["eta"] * 0.5
    S = inp["S"].cuda()
    S_ref = inp["S"].double().numpy()
    tol = TOL[inp["q"].dtype]
    for t in range(5):
        a = None if not decay else inp["alpha"][t]
        g = {n: inp[n][t].cuda() for n in ("q", "k", "v", "eta")}
        o = kla.kla_decode_step(g["q"], g["k"], g["v"], None if a is None else a.cuda(), g["eta"],
                                inp["eps"], S, beta_mode=mode)
        o_ref, S_ref = oracle.decode(inp["q"][t], inp["k"][t], inp["v"][t], a, inp["eta"][t],
                                     inp["eps"], S_ref, beta_mode=mode)
        torch.cuda.synchronize()
        assert rel_err(o, o_ref) <= tol
        assert rel_err(S, S_ref) <= tol


def test_given_mode_with_kaczmarz_coefficient_matches_kaczmarz_mode():
    """On the GPU too: beta precomputed as eta/(||k||^2+eps) (fp32, torch)
    and passed as the given beta reproduces the Kaczmarz mode."""
    inp = prefill_inputs(1, 256, 2, 128, 128, "bf16", seed=95, s0_var=0.01)
    d = cuda(inp)
    n2 = (d["k"].float() ** 2).sum(-1)
    beta = d["eta"] / (n2 + d["eps"])
    o1, S1 = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"], d["S0"])
    o2, S2 = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], beta.contiguous(), d["eps"],
                               d["S0"], beta_mode="given")
    torch.cuda.synchronize()
    assert rel_err(o2.float(), o1.float().cpu().double().numpy()) <= 1e-2
    assert rel_err(S2, S1.cpu().double().numpy()) <= 1e-2
