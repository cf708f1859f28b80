"""GPU parity of kla_decode_step and kla_chunk_fwd_varlen against the fp64
oracle (max abs error / max |oracle| per tensor: 1e-4 fp32, 2e-2 bf16)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300.workloads import (WORKLOADS, decode_inputs, prefill_inputs,
                                                       varlen_inputs)
from tests._util import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,dtype", [(64, "fp32"), (128, "fp32"), (64, "bf16"), (128, "bf16")])
def test_decode_steps_small(d, dtype):
    inp = decode_inputs(3, 5, d, d, steps=6, dtype=dtype, seed=20 + d)
    S = inp["S"].cuda()
    S_ref = inp["S"].double().numpy()
    tol = TOL[inp["q"].dtype]
    for t in range(6):
        g = {n: inp[n][t].cuda() for n in ("q", "k", "v", "alpha", "eta")}
        o = kla.kla_decode_step(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], S)
        o_ref, S_ref = oracle.decode(inp["q"][t], inp["k"][t], inp["v"][t], inp["alpha"][t],
                                     inp["eta"][t], inp["eps"], S_ref)
        torch.cuda.synchronize()
        assert o.dtype == inp["q"].dtype
        assert rel_err(o, o_ref) <= tol
        assert rel_err(S, S_ref) <= tol


def test_decode_full_size_sampled_units():
    """B=256 H=16 d=128, 64 steps in place (the timed decode workload); the
    oracle follows 96 sampled (b, h) states through all 64 steps."""
    inp = WORKLOADS["decode_b256"].make()
    steps = inp["q"].shape[0]
    S = inp["S"].cuda()
    rng = np.random.default_rng(0)
    units = rng.choice(256 * 16, size=96, replace=False)
    bi, hi = units // 16, units % 16
    S_ref = inp["S"][bi, hi].double().numpy()[:, None]        # [96,1,d,d]
    errs_o = []
    outs = []
    for t in range(steps):
        g = {n: inp[n][t].cuda() for n in ("q", "k", "v", "alpha", "eta")}
        outs.append(kla.kla_decode_step(g["q"], g["k"], g["v"], g["alpha"], g["eta"],
                                        inp["eps"], S))
    torch.cuda.synchronize()
    o_all_ref = []
    for t in range(steps):
        sel = lambda x: x[t][bi, hi][:, None]
        o_ref, S_ref = oracle.decode(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]),
                                     sel(inp["alpha"]), sel(inp["eta"]), inp["eps"], S_ref,
                                     nthreads=8)
        o_all_ref.append(o_ref[:, 0])
    o_gpu = torch.stack([o[bi, hi] for o in outs])
    assert rel_err(o_gpu, np.stack(o_all_ref)) <= 2e-2
    assert rel_err(S[bi, hi], S_ref[:, 0]) <= 2e-2


def test_decode_steps_equal_prefill():
    """64 decode steps from S0 give the same outputs and state as one prefill
    over the same 64 tokens."""
    inp = prefill_inputs(2, 64, 3, 128, 128, "fp32", seed=30, s0_var=0.01)
    d = cuda(inp)
    o_p, S_p = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"], d["S0"])
    S = d["S0"].clone()
    outs = []
    for t in range(64):
        outs.append(kla.kla_decode_step(d["q"][:, t].contiguous(), d["k"][:, t].contiguous(),
                                        d["v"][:, t].contiguous(), d["alpha"][:, t].contiguous(),
                                        d["eta"][:, t].contiguous(), d["eps"], S))
    torch.cuda.synchronize()
    o_d = torch.stack(outs, 1)
    assert rel_err(o_d, o_p.cpu().double().numpy()) <= 1e-4
    assert rel_err(S, S_p.cpu().double().numpy()) <= 1e-4


def _varlen(inp, **kw):
    d = cuda(inp)
    return kla.kla_chunk_fwd_varlen(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"],
                                    d["cu_seqlens"], d["S0"], check_status=True, **kw)


@pytest.mark.parametrize("d,dtype", [(64, "fp32"), (128, "fp32"), (128, "bf16"), (64, "bf16")])
def test_varlen_small(d, dtype):
    lens = [1, 63, 64, 65, 0, 130, 7, 200]
    inp = varlen_inputs(lens, 2, d, d, dtype, seed=40 + d, s0_var=0.01)
    o, S = _varlen(inp)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_varlen(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                         inp["eps"], inp["cu_seqlens"], inp["S0"], nthreads=8)
    tol = TOL[inp["q"].dtype]
    assert rel_err(o, o_ref) <= tol
    assert rel_err(S, S_ref) <= tol


def test_varlen_equals_per_sequence_calls():
    lens = [70, 5, 128, 191]
    inp = varlen_inputs(lens, 2, 128, 128, "bf16", seed=50, s0_var=0.01)
    o, S = _varlen(inp)
    cu = inp["cu_seqlens"].tolist()
    d = cuda(inp)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        o1, S1 = kla.kla_chunk_fwd(d["q"][None, a:b].contiguous(), d["k"][None, a:b].contiguous(),
                                   d["v"][None, a:b].contiguous(), d["alpha"][None, a:b].contiguous(),
                                   d["eta"][None, a:b].contiguous(), d["eps"], d["S0"][n:n + 1])
        torch.cuda.synchronize()
        # a sequence shorter than one chunk runs on the fp32 CUDA-core kernel when
        # called alone, so the two results agree to the bf16 tolerance, not bitwise
        assert rel_err(o[a:b], o1[0].cpu().double().numpy()) <= 2e-2
        assert rel_err(S[n], S1[0].cpu().double().numpy()) <= 2e-2
        if b - a >= 64:
            torch.testing.assert_close(S[n], S1[0], rtol=0, atol=0)
            torch.testing.assert_close(o[a:b], o1[0], rtol=0, atol=0)


@pytest.mark.parametrize("bad", ["decreasing", "first_nonzero", "last_mismatch"])
def test_varlen_bad_seqlens_reported_by_device(bad):
    lens = [10, 20, 30]
    inp = varlen_inputs(lens, 2, 64, 64, "fp32", seed=60)
    cu = inp["cu_seqlens"].clone()
    if bad == "decreasing":
        cu[1], cu[2] = 25, 12
    elif bad == "first_nonzero":
        cu[0] = 3
    else:
        cu[-1] = 50      # total_T is 60
    inp["cu_seqlens"] = cu
    with pytest.raises(kla.KlaError) as ei:
        _varlen(inp)
    assert ei.value.status == 1


def test_varlen_full_size_sampled():
    """64 sequences, lengths U[128, 8192], H=16 d=128 bf16: the GPU runs the
    packed batch; the oracle recomputes 6 sampled sequences on 3 heads."""
    inp = WORKLOADS["varlen_64"].make()
    o, S = _varlen(inp)
    torch.cuda.synchronize()
    cu = inp["cu_seqlens"].numpy()
    rng = np.random.default_rng(1)
    seqs = sorted(rng.choice(64, size=6, replace=False).tolist())
    heads = [0, 7, 15]
    for n in seqs:
        a, b = int(cu[n]), int(cu[n + 1])
        sel = lambda x: x[a:b][:, heads][None].contiguous()
        o_ref, S_ref = oracle.forward(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]),
                                      sel(inp["alpha"]), sel(inp["eta"]), inp["eps"],
                                      inp["S0"][n:n + 1, heads], nthreads=3)
        assert rel_err(o[a:b][:, heads], o_ref[0]) <= 2e-2
        assert rel_err(S[n, heads], S_ref[0]) <= 2e-2
