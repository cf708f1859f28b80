"""GPU parity of the wide state pass (one 128-column CTA per (sequence,
head) in the two-launch forward, chosen when two 64-column CTAs per head
would outnumber the SMs) against the fp64 oracle, error max|gpu - oracle| /
max|oracle| <= 2e-2 (bf16).  KLA_WIDE_STATE=1 forces it on small cases; the
forward, the varlen forward and the backward's state recording run through
it."""
import numpy as np
import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300.workloads import prefill_inputs, varlen_inputs
from tests._util import cuda, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture
def wide(monkeypatch):
    def set_w(on):
        monkeypatch.setenv("KLA_WIDE_STATE", "1" if on else "0")
    return set_w


# an odd number of chunks per sequence keeps the fixed-length forward on the
# two-launch path (phase 1, then the state pass)
@pytest.mark.parametrize("B,T,H,with_S0,no_alpha,mode", [
    (2, 448, 3, True, False, "kaczmarz"), (1, 320, 2, False, False, "kaczmarz"),
    (3, 64, 2, True, True, "given"), (2, 130, 2, True, False, "kaczmarz")])
def test_wide_forward_parity(wide, B, T, H, with_S0, no_alpha, mode):
    wide(True)
    inp = prefill_inputs(B, T, H, 128, 128, "bf16", seed=700 + T, s0_var=0.01)
    g = cuda(inp)
    n0 = kla.kla_launch_count()
    o, S = kla.kla_chunk_fwd(g["q"], g["k"], g["v"], None if no_alpha else g["alpha"], g["eta"],
                             inp["eps"], g["S0"] if with_S0 else None, beta_mode=mode)
    torch.cuda.synchronize()
    if ((T + 63) // 64) % 2 == 1:
        assert kla.kla_launch_count() - n0 == 2
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"], None if no_alpha else inp["alpha"],
                                  inp["eta"], inp["eps"], inp["S0"] if with_S0 else None,
                                  nthreads=8, beta_mode=mode)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2


def test_wide_matches_narrow(wide):
    """The wide and the narrow state pass compute the same products."""
    inp = prefill_inputs(2, 448, 2, 128, 128, "bf16", seed=71, s0_var=0.01)
    g = cuda(inp)
    args = (g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"])
    wide(False)
    o0, S0 = kla.kla_chunk_fwd(*args)
    wide(True)
    o1, S1 = kla.kla_chunk_fwd(*args)
    torch.cuda.synchronize()
    assert rel_err(o1, o0.double().cpu().numpy()) <= 1e-3
    assert rel_err(S1, S0.double().cpu().numpy()) <= 1e-5


def test_wide_varlen_parity(wide):
    wide(True)
    lens = [1, 63, 64, 65, 0, 130, 7, 200]
    inp = varlen_inputs(lens, 2, 128, 128, "bf16", seed=72, s0_var=0.01)
    d = cuda(inp)
    n0 = kla.kla_launch_count()
    o, S = kla.kla_chunk_fwd_varlen(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"],
                                    d["cu_seqlens"], d["S0"], check_status=True)
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == 3   # prep, phase 1, state pass
    o_ref, S_ref = oracle.forward_varlen(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                         inp["eps"], inp["cu_seqlens"], inp["S0"], nthreads=8)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2


def test_wide_backward_parity(wide):
    """The backward's forward records the chunk-start states through the wide pass."""
    wide(True)
    B, T, H, d = 2, 200, 2, 128
    inp = prefill_inputs(B, T, H, d, d, "bf16", seed=73, s0_var=0.01)
    rng = np.random.default_rng(74)
    do = torch.from_numpy(rng.standard_normal((B, T, H, d)).astype(np.float32)).to(torch.bfloat16)
    dST = torch.from_numpy((0.1 * rng.standard_normal((B, H, d, d))).astype(np.float32))
    g = cuda(dict(inp, do=do, dST=dST))
    got = kla.kla_chunk_bwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"],
                            g["do"], g["dST"])
    torch.cuda.synchronize()
    ref = oracle.backward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"], inp["eps"],
                          inp["S0"], do, dST, nthreads=8)
    for name, a, b in zip(("dq", "dk", "dv", "dalpha", "deta", "dS0"), got, ref):
        assert rel_err(a, b) <= 2e-2, name
