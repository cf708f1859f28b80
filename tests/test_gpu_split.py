"""GPU parity of the sequence-split forward (fixed-length batches run as P
segments per sequence: the state pass of each segment from a zero state, the
transition pass of the later segments from the identity, the segment start
states combined in order and the later segments' outputs corrected) against
the fp64 oracle, error max|gpu - oracle| / max|oracle| <= 2e-2 (bf16).  The
split factor is forced through KLA_SEQ_SPLIT for the small cases; the
long-context workload (B1 H16 T32768) takes it by default."""
import os

import numpy as np
import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300.workloads import prefill_inputs
from tests._util import cuda, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture
def split(monkeypatch):
    def set_p(P):
        monkeypatch.setenv("KLA_SEQ_SPLIT", str(P))
    return set_p


# launches: the fused launch (phase 1, state and transition passes) when the
# state and transition CTAs fit on half of the SMs, else phase 1 and the state
# + transition launch; then the combine and the correction
@pytest.mark.parametrize("B,T,H,P,with_S0,no_alpha,mode,launches", [
    (1, 512, 2, 2, True, False, "kaczmarz", 3), (2, 512, 2, 4, True, False, "kaczmarz", 3),
    (2, 768, 3, 3, False, False, "kaczmarz", 3), (1, 1024, 2, 8, True, True, "kaczmarz", 3),
    (2, 256, 2, 2, True, False, "given", 3), (4, 1024, 8, 2, True, False, "kaczmarz", 4)])
def test_split_forward_parity(split, B, T, H, P, with_S0, no_alpha, mode, launches):
    split(P)
    inp = prefill_inputs(B, T, H, 128, 128, "bf16", seed=400 + T + P, s0_var=0.01)
    g = cuda(inp)
    S0 = inp["S0"] if with_S0 else None
    n0 = kla.kla_launch_count()
    o, S = kla.kla_chunk_fwd(g["q"], g["k"], g["v"], None if no_alpha else g["alpha"], g["eta"],
                             inp["eps"], g["S0"] if with_S0 else None, beta_mode=mode)
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == launches
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"], None if no_alpha else inp["alpha"],
                                  inp["eta"], inp["eps"], S0, nthreads=8, beta_mode=mode)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2


@pytest.mark.parametrize("B,T,H,P,with_S0,no_alpha,mode", [
    (1, 4096, 16, 4, True, False, "kaczmarz"),   # 16 x 7 chains: two CTAs each would not fit
    (2, 2048, 16, 2, False, True, "given"),      # 32 x 3 chains
])
def test_split_with_one_wide_cta_per_chain(split, B, T, H, P, with_S0, no_alpha, mode):
    """A split whose state and transition chains in two 64-column CTAs each
    would outnumber the SMs runs one 128-column CTA per chain: phase 1, the
    state and transition launch, the combine and the correction."""
    split(P)
    inp = prefill_inputs(B, T, H, 128, 128, "bf16", seed=500 + T + P, s0_var=0.01)
    g = cuda(inp)
    S0 = inp["S0"] if with_S0 else None
    n0 = kla.kla_launch_count()
    o, S = kla.kla_chunk_fwd(g["q"], g["k"], g["v"], None if no_alpha else g["alpha"], g["eta"],
                             inp["eps"], g["S0"] if with_S0 else None, beta_mode=mode)
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == 4
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"], None if no_alpha else inp["alpha"],
                                  inp["eta"], inp["eps"], S0, nthreads=16, beta_mode=mode)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2


def test_split_matches_unsplit(split):
    """The split and the fused single-chain forward agree (both bf16 paths)."""
    inp = prefill_inputs(2, 1024, 2, 128, 128, "bf16", seed=9, s0_var=0.01)
    g = cuda(inp)
    args = (g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"])
    split(1)
    o1, S1 = kla.kla_chunk_fwd(*args)
    split(4)
    o4, S4 = kla.kla_chunk_fwd(*args)
    torch.cuda.synchronize()
    assert rel_err(o4, o1.double().cpu().numpy()) <= 2e-2
    assert rel_err(S4, S1.double().cpu().numpy()) <= 2e-2


def test_split_invalid_factor_falls_back(split):
    """A factor whose segments are not whole 128-token tiles runs unsplit."""
    split(3)
    inp = prefill_inputs(1, 512, 2, 128, 128, "bf16", seed=10)
    g = cuda(inp)
    n0 = kla.kla_launch_count()
    o, S = kla.kla_chunk_fwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"])
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == 1   # the fused launch
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                  inp["eps"], inp["S0"], nthreads=8)
    assert rel_err(o, o_ref) <= 2e-2


def test_long_context_takes_the_split_sampled(monkeypatch):
    """long_context (B1 H16 T32768 d128 bf16) runs split by default; two heads
    checked against the oracle run on those heads alone."""
    monkeypatch.delenv("KLA_SEQ_SPLIT", raising=False)
    from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS
    wl = WORKLOADS["long_context"]
    inp = wl.make()
    g = cuda(inp)
    n0 = kla.kla_launch_count()
    o, S = kla.kla_chunk_fwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], wl.eps, g["S0"])
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == 4   # phase 1, state + transition, combine, correct
    for h in (0, 11):
        sl = lambda x: x[:, :, h:h + 1].contiguous()
        o_ref, S_ref = oracle.forward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["alpha"]),
                                      sl(inp["eta"]), wl.eps,
                                      None if inp["S0"] is None else inp["S0"][:, h:h + 1])
        assert rel_err(o[:, :, h:h + 1], o_ref) <= 2e-2
        assert rel_err(S[:, h:h + 1], S_ref) <= 2e-2
