"""GPU parity of the backward pass (kla_chunk_bwd) against the fp64 backward
oracle: every gradient (dq, dk, dv, dalpha, deta, dS0) element by element,
error max|gpu - oracle| / max|oracle| within 1e-4 (fp32) and 2e-2 (bf16)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300.workloads import prefill_inputs
from tests._util import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu


def _grad_inputs(B, T, H, d, dtype, seed):
    rng = np.random.default_rng(seed)
    t = torch.bfloat16 if dtype == "bf16" else torch.float32
    do = torch.from_numpy(rng.standard_normal((B, T, H, d)).astype(np.float32)).to(t)
    dST = torch.from_numpy((0.1 * rng.standard_normal((B, H, d, d))).astype(np.float32))
    return do, dST


def _check(g, ref, tol, names=("dq", "dk", "dv", "dalpha", "deta", "dS0")):
    for n, a, b in zip(names, g, ref):
        if b is None:
            assert a is None, n
            continue
        e = rel_err(a, b)
        assert e <= tol, f"{n}: {e:.3e} > {tol}"


@pytest.mark.parametrize("B,T,H,d,dtype,mode,no_alpha,with_dST,with_S0", [
    (1, 256, 2, 64, "fp32", "kaczmarz", False, True, True),
    (2, 130, 2, 128, "fp32", "kaczmarz", False, True, True),
    (1, 77, 3, 64, "fp32", "given", False, False, True),
    (2, 64, 2, 128, "fp32", "kaczmarz", True, True, False),
    (2, 200, 2, 128, "bf16", "kaczmarz", False, True, True),
    (1, 320, 2, 128, "bf16", "given", False, True, False),
    (3, 5, 2, 64, "bf16", "kaczmarz", False, False, True)])
def test_backward_parity(B, T, H, d, dtype, mode, no_alpha, with_dST, with_S0):
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=200 + T, s0_var=0.01)
    do, dST = _grad_inputs(B, T, H, d, dtype, 300 + T)
    alpha = None if no_alpha else inp["alpha"]
    S0 = inp["S0"] if with_S0 else None
    dST = dST if with_dST else None
    g = cuda(dict(inp, do=do, dST=dST))
    got = kla.kla_chunk_bwd(g["q"], g["k"], g["v"], None if no_alpha else g["alpha"], g["eta"],
                            inp["eps"], g["S0"] if with_S0 else None, g["do"],
                            g["dST"] if with_dST else None, beta_mode=mode)
    torch.cuda.synchronize()
    ref = oracle.backward(inp["q"], inp["k"], inp["v"], alpha, inp["eta"], inp["eps"], S0, do,
                          dST, nthreads=8, beta_mode=mode)
    _check(got, ref, TOL[inp["q"].dtype])


def test_backward_launches_and_status():
    """Launch count of the bf16 d128 backward and a clean status word."""
    B, T, H, d = 2, 192, 2, 128
    inp = prefill_inputs(B, T, H, d, d, "bf16", seed=5)
    do, dST = _grad_inputs(B, T, H, d, "bf16", 6)
    g = cuda(dict(inp, do=do, dST=dST))
    ws = torch.zeros(kla.kla_chunk_bwd_workspace_size(B, T, H, d), dtype=torch.uint8,
                     device="cuda")
    args = (g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"], g["do"], g["dST"])
    kla.kla_chunk_bwd(*args, workspace=ws)
    torch.cuda.synchronize()
    n0 = kla.kla_launch_count()
    kla.kla_chunk_bwd(*args, workspace=ws)
    torch.cuda.synchronize()
    # bf16, d 128: the tensor-core forward recording the chunk-start states
    # (phase 1, state pass), the dS chain over its chunk workspace, the token
    # gradients
    assert kla.kla_launch_count() - n0 == 4
    assert kla.kla_workspace_status(ws) == 0


def test_backward_no_tokens_passes_the_state_gradient():
    B, H, d = 2, 2, 64
    q = torch.zeros((B, 0, H, d), device="cuda")
    eta = torch.zeros((B, 0, H), device="cuda")
    dST = torch.randn((B, H, d, d), device="cuda")
    _, _, _, _, _, dS0 = kla.kla_chunk_bwd(q, q, q, eta, eta, 1e-6, None, q, dST)
    torch.cuda.synchronize()
    assert torch.equal(dS0, dST)


def test_backward_full_size_sampled():
    """The layer workload (B4 H8 T2048 d128 bf16): all gradients of two sampled
    (batch, head) units against the oracle run on those units alone."""
    from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS
    wl = WORKLOADS["layer_prefill"]
    inp = wl.make()
    do, dST = _grad_inputs(wl.B, wl.T, wl.H, wl.d, "bf16", 7)
    g = cuda(dict(inp, do=do, dST=dST))
    got = kla.kla_chunk_bwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], wl.eps, g["S0"],
                            g["do"], g["dST"])
    torch.cuda.synchronize()
    for b, h in ((0, 0), (3, 5)):
        tok = lambda x: x[b:b + 1, :, h:h + 1].contiguous()
        st = lambda x: x[b:b + 1, h:h + 1].contiguous()
        ref = oracle.backward(tok(inp["q"]), tok(inp["k"]), tok(inp["v"]), tok(inp["alpha"]),
                              tok(inp["eta"]), wl.eps, st(inp["S0"]), tok(do), st(dST))
        sub = [tok(got[0]), tok(got[1]), tok(got[2]), tok(got[3]), tok(got[4]), st(got[5])]
        _check(sub, ref, TOL[torch.bfloat16])


def test_backward_cuda_core_launches():
    """fp32 (and d 64) take the CUDA-core forward for the states: three launches."""
    B, T, H, d = 1, 128, 2, 64
    inp = prefill_inputs(B, T, H, d, d, "fp32", seed=12)
    do, dST = _grad_inputs(B, T, H, d, "fp32", 13)
    g = cuda(dict(inp, do=do, dST=dST))
    args = (g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"], g["do"], g["dST"])
    kla.kla_chunk_bwd(*args)
    torch.cuda.synchronize()
    n0 = kla.kla_launch_count()
    kla.kla_chunk_bwd(*args)
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == 3


def _varlen_oracle_backward(inp, do, dST, mode="kaczmarz"):
    """The backward oracle run sequence by sequence on the packed inputs."""
    cu = inp["cu_seqlens"].tolist()
    N = len(cu) - 1
    outs = [np.zeros(inp["q"].shape), np.zeros(inp["k"].shape), np.zeros(inp["v"].shape),
            np.zeros(inp["alpha"].shape), np.zeros(inp["eta"].shape),
            np.zeros(inp["S0"].shape if inp["S0"] is not None else dST.shape)]
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        sl = lambda x: x[None, a:b]
        S0 = None if inp["S0"] is None else inp["S0"][n:n + 1]
        g = oracle.backward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["alpha"]),
                            sl(inp["eta"]), inp["eps"], S0, sl(do), dST[n:n + 1], beta_mode=mode)
        for i in range(5):
            outs[i][a:b] = g[i][0]
        outs[5][n] = g[5][0]
    return outs


@pytest.mark.parametrize("d,dtype,mode", [(128, "bf16", "kaczmarz"), (64, "fp32", "kaczmarz"),
                                          (128, "bf16", "given")])
def test_varlen_backward_parity(d, dtype, mode):
    """Packed sequences (an empty one, shorter than a chunk, exact multiples,
    ragged) against the oracle per sequence."""
    from gated_delta_rule_kaczmarz_gb300.workloads import varlen_inputs
    lens = [70, 0, 5, 128, 191, 64]
    inp = varlen_inputs(lens, 2, d, d, dtype, seed=60 + d, s0_var=0.01)
    rng = np.random.default_rng(61)
    total = sum(lens)
    t = torch.bfloat16 if dtype == "bf16" else torch.float32
    do = torch.from_numpy(rng.standard_normal((total, 2, d)).astype(np.float32)).to(t)
    dST = torch.from_numpy((0.1 * rng.standard_normal((len(lens), 2, d, d))).astype(np.float32))
    g = cuda(dict(inp, do=do, dST=dST))
    got = kla.kla_chunk_bwd_varlen(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"],
                                   g["cu_seqlens"], g["S0"], g["do"], g["dST"], beta_mode=mode)
    torch.cuda.synchronize()
    ref = _varlen_oracle_backward(inp, do, dST, mode)
    _check(got, ref, TOL[t])


def test_varlen_backward_bad_seqlens_reported():
    """A decreasing cu_seqlens is caught on the device; the status word says so."""
    from gated_delta_rule_kaczmarz_gb300.workloads import varlen_inputs
    inp = varlen_inputs([64, 64], 2, 128, 128, "bf16", seed=62)
    g = cuda(inp)
    cu = torch.tensor([0, 100, 64], dtype=torch.int32, device="cuda")   # not non-decreasing
    do = torch.zeros_like(g["v"])
    ws = torch.zeros(kla.kla_chunk_bwd_varlen_workspace_size(2, 128, 2, 128, 1),
                     dtype=torch.uint8, device="cuda")
    kla.kla_chunk_bwd_varlen(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], cu, None,
                             do, workspace=ws)
    with pytest.raises(kla.KlaError) as ei:
        kla.kla_workspace_status(ws)
    assert ei.value.status == kla.binding.KLA_ERR_INVALID_ARG


@pytest.mark.parametrize("B,T,H,d,dtype", [
    (1, 64, 1, 128, "bf16"),    # exactly one chunk, tensor-core states
    (1, 65, 1, 128, "bf16"),    # one row into the second chunk
    (3, 20, 1, 128, "bf16"),    # B*T < 64: CUDA-core states for bf16 d 128
    (2, 127, 3, 64, "bf16")])   # d 64 bf16
def test_backward_edge_shapes(B, T, H, d, dtype):
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=700 + T, s0_var=0.01)
    do, dST = _grad_inputs(B, T, H, d, dtype, 701 + T)
    g = cuda(dict(inp, do=do, dST=dST))
    got = kla.kla_chunk_bwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"],
                            g["do"], g["dST"])
    torch.cuda.synchronize()
    ref = oracle.backward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"], inp["eps"],
                          inp["S0"], do, dST)
    _check(got, ref, TOL[inp["q"].dtype])
