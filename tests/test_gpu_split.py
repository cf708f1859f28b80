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
# segments are equal and the state and transition CTAs fit on half of the
# SMs, else phase 1 and the state + transition launch; then the combine and
# the correction.  Segments are whole 128-token tiles, as equal as the tile
# count allows (640 tokens in 2: 3 + 2 tiles; 896 in 3: 3 + 2 + 2; 512 in 3:
# 2 + 1 + 1; 1152 in 8: 2 + 1 x 7).
@pytest.mark.parametrize("B,T,H,P,with_S0,no_alpha,mode,launches", [
    (1, 512, 2, 2, True, False, "kaczmarz", 3), (2, 512, 2, 4, True, False, "kaczmarz", 3),
    (2, 768, 3, 3, False, False, "kaczmarz", 3), (1, 1024, 2, 8, True, True, "kaczmarz", 3),
    (2, 256, 2, 2, True, False, "given", 3), (4, 1024, 8, 2, True, False, "kaczmarz", 4),
    (1, 640, 2, 2, True, False, "kaczmarz", 4), (2, 896, 3, 3, True, True, "kaczmarz", 4),
    (1, 512, 2, 3, False, False, "given", 4), (1, 1152, 2, 8, True, False, "kaczmarz", 4)])
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
    (1, 4608, 16, 5, True, False, "kaczmarz"),   # 16 x 9 chains, segments of 8 + 7 x 4 tiles
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
    """A factor above the sequence's count of 128-token tiles runs unsplit."""
    split(5)
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


def _unequal_draws(n, seed):
    """Seeded shapes whose forced factor leaves segments of unequal length:
    T a whole number of 128-token tiles (2 to 12), P from 2 to min(8, tiles)
    not dividing it."""
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        tiles = int(rng.integers(2, 13))
        P = int(rng.integers(2, min(8, tiles) + 1))
        if tiles % P == 0:
            continue
        cases.append(dict(B=int(rng.integers(1, 4)), T=128 * tiles, H=int(rng.integers(1, 5)),
                          P=P, s0=float(rng.choice([0.0, 0.01])), seed=int(rng.integers(1 << 30))))
    return cases


UNEQUAL = _unequal_draws(6, 20261203)


@pytest.mark.parametrize("case", UNEQUAL, ids=[f"unequal{i}" for i in range(len(UNEQUAL))])
def test_split_unequal_segments_random(split, case):
    c = case
    split(c["P"])
    inp = prefill_inputs(c["B"], c["T"], c["H"], 128, 128, "bf16", seed=c["seed"], s0_var=c["s0"])
    g = cuda(inp)
    n0 = kla.kla_launch_count()
    o, S = kla.kla_chunk_fwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"])
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == 4   # phase 1, state + transition, combine, correction
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                  inp["eps"], inp["S0"], nthreads=8)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2
