"""GPU parity of the chunkwise prefill (kla_chunk_fwd) against the fp64 oracle.

Every comparison is element by element on the same seeded inputs; the error
measure is max|gpu - oracle| / max|oracle| per output tensor, bounded by 1e-4
for fp32 inputs and 2e-2 for bf16 inputs (fp32 state)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS, prefill_inputs
from tests._util import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu


def _run(inp):
    d = cuda(inp)
    o, S = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"], d["S0"])
    torch.cuda.synchronize()
    return o, S


def _oracle(inp, nthreads=8):
    return oracle.forward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"], inp["eps"],
                          inp["S0"], nthreads=nthreads)


def test_tiny_fp32_workload():
    """B=1 H=2 T=256 d=64 fp32, S0 = 0: the fp32 parity case at 1e-4."""
    inp = WORKLOADS["tiny_fp32"].make()
    o, S = _run(inp)
    o_ref, S_ref = _oracle(inp)
    assert rel_err(o, o_ref) <= 1e-4
    assert rel_err(S, S_ref) <= 1e-4


CASES = [
    # B, T, H, d, dtype, key_norm_sigma, s0_var
    (2, 200, 3, 64, "fp32", 0.5, 0.01),     # ragged tail, several chunks
    (1, 1, 2, 128, "fp32", 0.5, 0.01),      # single token
    (2, 63, 2, 128, "fp32", 1.0, 0.0),      # one partial chunk
    (1, 65, 2, 128, "fp32", 0.5, 0.01),     # chunk + 1
    (3, 130, 2, 64, "bf16", 0.5, 0.01),
    (2, 257, 4, 128, "bf16", 0.5, 0.01),
    (1, 500, 2, 128, "bf16", 1.0, 0.0),     # lognormal(0,1) key norms
    (2, 64, 2, 128, "bf16", 0.5, 0.0),
    (1, 1, 2, 128, "bf16", 0.5, 0.01),      # fewer tokens than one chunk in total
    (2, 63, 3, 128, "bf16", 0.5, 0.01),     # partial chunks only
    (1, 65, 2, 128, "bf16", 1.0, 0.01),
    (3, 129, 2, 128, "bf16", 0.5, 0.0),     # odd number of chunks per CTA pair
    (1, 1000, 1, 128, "bf16", 1.0, 0.01),
]


@pytest.mark.parametrize("B,T,H,d,dtype,sig,s0", CASES)
def test_parity_small(B, T, H, d, dtype, sig, s0):
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=100 + T, key_norm_sigma=sig, s0_var=s0)
    o, S = _run(inp)
    o_ref, S_ref = _oracle(inp)
    tol = TOL[inp["q"].dtype]
    assert o.dtype == inp["q"].dtype
    assert rel_err(o, o_ref) <= tol
    assert rel_err(S, S_ref) <= tol


@pytest.mark.parametrize("varlen", [False, True])
def test_bf16_d128_runs_on_the_tensor_core_kernels(varlen):
    """bf16 with d = 128 takes the tcgen05 path.  A fixed-length batch with an
    even number of chunks per sequence and a small state pass is one fused
    launch (phase 1 and the state pass together); varlen is a sequence-table
    launch, the intra-chunk launch and the state-pass launch."""
    inp = prefill_inputs(2, 256, 2, 128, 128, "bf16", seed=11, s0_var=0.01)
    d = cuda(inp)
    n0 = kla.kla_launch_count()
    if varlen:
        cu = torch.tensor([0, 256, 512], dtype=torch.int32, device="cuda")
        f = lambda x: x.reshape(512, *x.shape[2:])
        kla.kla_chunk_fwd_varlen(f(d["q"]), f(d["k"]), f(d["v"]), f(d["alpha"]), f(d["eta"]),
                                 d["eps"], cu, d["S0"])
    else:
        kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"], d["S0"])
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == (3 if varlen else 1)
    ws = kla.kla_chunk_fwd_workspace_size(2, 256, 2, 128, 128)
    assert ws > 256


def test_odd_chunk_count_uses_two_launches():
    """Three chunks per sequence: the intra-chunk and state-pass launches."""
    inp = prefill_inputs(1, 129, 2, 128, 128, "bf16", seed=12, s0_var=0.01)
    d = cuda(inp)
    n0 = kla.kla_launch_count()
    kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"], d["S0"])
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == 2


def test_fused_launch_equals_two_launch_path():
    """Sequences of a batch are independent: 48 sequences x 2 heads (too many
    state-pass CTAs for the fused launch: two launches) give bitwise the same
    outputs and states as the same sequences in batches of 4 (fused launch)."""
    inp = prefill_inputs(48, 128, 2, 128, 128, "bf16", seed=13, s0_var=0.01)
    d = cuda(inp)
    n0 = kla.kla_launch_count()
    o_all, S_all = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"],
                                     d["S0"])
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == 2
    for b0 in range(0, 48, 4):
        sl = lambda x: x[b0:b0 + 4].contiguous()
        n1 = kla.kla_launch_count()
        o, S = kla.kla_chunk_fwd(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["alpha"]), sl(d["eta"]),
                                 d["eps"], sl(d["S0"]))
        torch.cuda.synchronize()
        assert kla.kla_launch_count() - n1 == 1
        torch.testing.assert_close(o, o_all[b0:b0 + 4], rtol=0, atol=0)
        torch.testing.assert_close(S, S_all[b0:b0 + 4], rtol=0, atol=0)


def test_eta_zero_is_pure_decay():
    """eta = 0: only the decay acts (alpha in [0.9, 1] keeps the product of
    150 decays inside the fp32 range)."""
    inp = prefill_inputs(1, 150, 2, 64, 64, "fp32", seed=5, s0_var=1.0)
    inp["eta"].zero_()
    inp["alpha"] = 0.9 + 0.1 * inp["alpha"]
    o, S = _run(inp)
    o_ref, S_ref = _oracle(inp)
    assert rel_err(o, o_ref) <= 1e-4 and rel_err(S, S_ref) <= 1e-4


def test_zero_length_writes_initial_state():
    inp = prefill_inputs(2, 0, 2, 64, 64, "fp32", seed=6, s0_var=1.0)
    o, S = _run(inp)
    assert o.numel() == 0
    torch.testing.assert_close(S.cpu(), inp["S0"], rtol=0, atol=0)
    inp["S0"] = None
    _, S = _run(inp)
    assert float(S.abs().max()) == 0.0


def test_in_place_state_and_no_final_state():
    inp = prefill_inputs(1, 100, 2, 128, 128, "bf16", seed=7, s0_var=0.01)
    d = cuda(inp)
    S = d["S0"].clone()
    o1, _ = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"], S, S_T=S)
    o2, none = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"], d["S0"],
                                 return_final_state=False)
    torch.cuda.synchronize()
    assert none is None
    o_ref, S_ref = _oracle(inp)
    assert rel_err(S, S_ref) <= 2e-2
    assert rel_err(o1, o_ref) <= 2e-2 and rel_err(o2, o_ref) <= 2e-2


@pytest.mark.parametrize("T1", [64, 100])
def test_split_and_resume_equals_one_call(T1):
    """fwd(x[:T1]) -> S, then fwd(x[T1:], S0=S) equals fwd(x): the state is the
    checkpoint, on and off a chunk boundary."""
    inp = prefill_inputs(2, 300, 2, 64, 64, "fp32", seed=8, s0_var=0.01)
    d = cuda(inp)
    o_full, S_full = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"], d["S0"])
    sl = lambda x, a, b: x[:, a:b].contiguous()
    o1, S1 = kla.kla_chunk_fwd(sl(d["q"], 0, T1), sl(d["k"], 0, T1), sl(d["v"], 0, T1),
                               sl(d["alpha"], 0, T1), sl(d["eta"], 0, T1), d["eps"], d["S0"])
    o2, S2 = kla.kla_chunk_fwd(sl(d["q"], T1, None), sl(d["k"], T1, None), sl(d["v"], T1, None),
                               sl(d["alpha"], T1, None), sl(d["eta"], T1, None), d["eps"], S1)
    torch.cuda.synchronize()
    o_ref, S_ref = _oracle(inp)
    assert rel_err(torch.cat([o1, o2], 1), o_ref) <= 1e-4
    assert rel_err(S2, S_ref) <= 1e-4
    assert rel_err(o_full, o_ref) <= 1e-4


def test_fp32_and_bf16_paths_agree():
    inp = prefill_inputs(1, 256, 2, 128, 128, "bf16", seed=9, s0_var=0.01)
    d = cuda(inp)
    o_b, S_b = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"], d["S0"])
    f = lambda x: x.float()
    o_f, S_f = kla.kla_chunk_fwd(f(d["q"]), f(d["k"]), f(d["v"]), d["alpha"], d["eta"], d["eps"],
                                 d["S0"])
    torch.cuda.synchronize()
    assert rel_err(o_b.float(), o_f.cpu().double().numpy()) <= 2e-2
    assert rel_err(S_b, S_f.cpu().double().numpy()) <= 2e-2


def test_layer_prefill_full_size():
    """B=4 H=8 T=2048 d=128 bf16, S0 ~ N(0,0.01): every output and state
    compared with the oracle (all 32 heads)."""
    inp = WORKLOADS["layer_prefill"].make()
    o, S = _run(inp)
    o_ref, S_ref = _oracle(inp, nthreads=16)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2


def test_long_context_full_size_sampled_heads():
    """B=1 H=16 T=32768 d=128 bf16, key norms lognormal(0,1), eta = 1: the GPU
    runs the whole problem; the oracle recomputes two sampled heads."""
    wl = WORKLOADS["long_context"]
    inp = wl.make()
    o, S = _run(inp)
    heads = [3, 12]
    sub = {n: (x[:, :, heads].contiguous() if n in ("q", "k", "v", "alpha", "eta") else x)
           for n, x in inp.items()}
    o_ref, S_ref = oracle.forward(sub["q"], sub["k"], sub["v"], sub["alpha"], sub["eta"],
                                  inp["eps"], None, nthreads=2)
    assert rel_err(o[:, :, heads], o_ref) <= 2e-2
    assert rel_err(S[:, heads], S_ref) <= 2e-2
