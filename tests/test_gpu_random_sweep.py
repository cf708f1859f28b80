"""Seeded random-shape sweep of the GPU entry points against the fp64 oracle.

The other GPU tests pick their shapes by hand (chunk and block boundaries,
edge values); this one draws them: batch sizes, sequence lengths (including
one-token, empty and ragged sequences), head counts, key-norm spreads,
initial states, write-coefficient modes and the no-decay case, for the
fixed-length forward on both kernel families and with the wide state pass or
the sequence split forced, the packed (varlen) forward on both families, the
decode step, the CCQ query, the backward and the no-allocation entry point.
Every draw comes from a fixed seed, so a
failure names a reproducible case.  Error measure and tolerances as in
tests/_util.py (max |gpu - oracle| / max |oracle| <= 2e-2 for bf16 inputs,
1e-4 for fp32); the device status word must read OK after every call."""
import numpy as np
import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300 import binding
from gated_delta_rule_kaczmarz_gb300.workloads import prefill_inputs, varlen_inputs
from tests._util import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu


def _draw_forward(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        bf16 = i % 4 != 3
        d = 128 if bf16 or rng.random() < 0.5 else 64
        cases.append(dict(B=int(rng.integers(1, 6)), T=int(rng.integers(1, 601)),
                          H=int(rng.integers(1, 7)), d=d, dtype="bf16" if bf16 else "fp32",
                          sigma=float(rng.choice([0.3, 0.5, 1.0])),
                          s0=float(rng.choice([0.0, 0.01])),
                          mode=str(rng.choice(["kaczmarz", "given"])),
                          no_alpha=bool(rng.random() < 0.2), seed=int(rng.integers(1 << 30))))
    return cases


def _draw_varlen(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        N = int(rng.integers(1, 9))
        lens = [int(x) for x in rng.integers(0, 401, N)]
        if N > 2:
            lens[int(rng.integers(N))] = 0                  # an empty sequence
            lens[int(rng.integers(N))] = 1                  # a one-token sequence
        cases.append(dict(lens=lens, H=int(rng.integers(1, 5)), s0=float(rng.choice([0.0, 0.01])),
                          seed=int(rng.integers(1 << 30))))
    return cases


FWD = _draw_forward(16, 20261203)
VARLEN = _draw_varlen(8, 20261204)


@pytest.mark.parametrize("case", FWD, ids=[f"fwd{i}" for i in range(len(FWD))])
def test_random_forward(case):
    c = case
    inp = prefill_inputs(c["B"], c["T"], c["H"], c["d"], c["d"], c["dtype"], seed=c["seed"],
                         key_norm_sigma=c["sigma"], s0_var=c["s0"])
    alpha = None if c["no_alpha"] else inp["alpha"]
    g = cuda(inp)
    dt = binding.KLA_DTYPE_BF16 if c["dtype"] == "bf16" else binding.KLA_DTYPE_F32
    nb = kla.kla_chunk_fwd_workspace_size(c["B"], c["T"], c["H"], c["d"], c["d"], dtype=dt)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    o, S = kla.kla_chunk_fwd(g["q"], g["k"], g["v"], None if alpha is None else g["alpha"],
                             g["eta"], inp["eps"], g["S0"], workspace=ws, beta_mode=c["mode"])
    assert kla.kla_workspace_status(ws) == binding.KLA_OK
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"], alpha, inp["eta"], inp["eps"],
                                  inp["S0"], nthreads=8, beta_mode=c["mode"])
    tol = TOL[inp["q"].dtype]
    assert rel_err(o, o_ref) <= tol
    assert rel_err(S, S_ref) <= tol


@pytest.mark.parametrize("case", VARLEN, ids=[f"varlen{i}" for i in range(len(VARLEN))])
def test_random_varlen(case):
    c = case
    inp = varlen_inputs(c["lens"], c["H"], 128, 128, "bf16", seed=c["seed"], s0_var=c["s0"])
    d = cuda(inp)
    o, S = kla.kla_chunk_fwd_varlen(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"],
                                    d["cu_seqlens"], d["S0"], check_status=True)
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_varlen(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                         inp["eps"], inp["cu_seqlens"], inp["S0"], nthreads=8)
    if sum(c["lens"]) > 0:
        assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2


def _lam(shape, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy((1.0 / (1.0 + np.exp(-rng.standard_normal(shape)))).astype(np.float32))


@pytest.mark.parametrize("seed", [31, 32, 33, 34])
def test_random_ccq_query(seed):
    rng = np.random.default_rng(seed)
    B, T, H = int(rng.integers(1, 5)), int(rng.integers(1, 501)), int(rng.integers(1, 5))
    inp = prefill_inputs(B, T, H, 128, 128, "bf16", seed=seed)
    lam = _lam((B, T, H), seed + 1)
    qc, (Ms, ms, ns) = kla.kla_ccq_query(cuda(inp)["q"], cuda(inp)["k"], lam.cuda())
    torch.cuda.synchronize()
    qc_ref, (Ms_ref, ms_ref, ns_ref) = oracle.ccq_query(inp["q"], inp["k"], lam, None)
    assert rel_err(qc, qc_ref) <= 2e-2, (B, T, H)
    assert rel_err(Ms, Ms_ref) <= 1e-5 and rel_err(ms, ms_ref) <= 1e-5
    assert np.array_equal(ns.cpu().numpy(), ns_ref)


@pytest.mark.parametrize("seed", [41, 42, 43])
def test_random_backward(seed):
    rng = np.random.default_rng(seed)
    bf16 = seed != 43
    d = 128 if bf16 else 64
    B, T, H = int(rng.integers(1, 4)), int(rng.integers(1, 201)), int(rng.integers(1, 4))
    dtype = "bf16" if bf16 else "fp32"
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=seed, s0_var=0.01)
    t = torch.bfloat16 if bf16 else torch.float32
    do = torch.from_numpy(rng.standard_normal((B, T, H, d)).astype(np.float32)).to(t)
    dST = torch.from_numpy((0.1 * rng.standard_normal((B, H, d, d))).astype(np.float32))
    g = cuda(dict(inp, do=do, dST=dST))
    got = kla.kla_chunk_bwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"],
                            g["do"], g["dST"])
    torch.cuda.synchronize()
    ref = oracle.backward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"], inp["eps"],
                          inp["S0"], do, dST, nthreads=8)
    tol = TOL[t]
    for name, a, b in zip(("dq", "dk", "dv", "dalpha", "deta", "dS0"), got, ref):
        assert rel_err(a, b) <= tol, (name, B, T, H, dtype)


def _forced_draws(n, seed):
    """Fixed-length bf16 cases run with a forced state-pass form: the wide
    (128-column) pass, or the sequence split into P segments."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        wide = i % 2 == 0
        cases.append(dict(B=int(rng.integers(1, 4)), T=int(rng.integers(64, 900)),
                          H=int(rng.integers(1, 4)), wide=wide,
                          P=0 if wide else int(rng.choice([2, 3, 4])),
                          s0=float(rng.choice([0.0, 0.01])), seed=int(rng.integers(1 << 30))))
    return cases


FORCED = _forced_draws(6, 20261205)


@pytest.mark.parametrize("case", FORCED, ids=[f"forced{i}" for i in range(len(FORCED))])
def test_random_forced_state_forms(monkeypatch, case):
    c = case
    if c["wide"]:
        monkeypatch.setenv("KLA_WIDE_STATE", "1")
    else:
        monkeypatch.setenv("KLA_SEQ_SPLIT", str(c["P"]))
    inp = prefill_inputs(c["B"], c["T"], c["H"], 128, 128, "bf16", seed=c["seed"], s0_var=c["s0"])
    g = cuda(inp)
    ws = torch.empty(kla.kla_chunk_fwd_workspace_size(c["B"], c["T"], c["H"], 128, 128),
                     dtype=torch.uint8, device="cuda")
    o, S = kla.kla_chunk_fwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"],
                             workspace=ws)
    assert kla.kla_workspace_status(ws) == binding.KLA_OK
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                  inp["eps"], inp["S0"], nthreads=8)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2


@pytest.mark.parametrize("seed", [51, 52, 53])
def test_random_varlen_fp32(seed):
    """Packed batches on the fp32 CUDA-core path (d = 64), with a workspace so
    that the device check of cu_seqlens runs and its status is read."""
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 7))
    lens = [int(x) for x in rng.integers(0, 300, N)]
    inp = varlen_inputs(lens, int(rng.integers(1, 4)), 64, 64, "fp32", seed=seed, s0_var=0.01)
    d = cuda(inp)
    o, S = kla.kla_chunk_fwd_varlen(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"],
                                    d["cu_seqlens"], d["S0"], check_status=True,
                                    workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.forward_varlen(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                         inp["eps"], inp["cu_seqlens"], inp["S0"], nthreads=8)
    if sum(lens) > 0:
        assert rel_err(o, o_ref) <= 1e-4
    assert rel_err(S, S_ref) <= 1e-4


@pytest.mark.parametrize("seed", [61, 62, 63, 64])
def test_random_decode(seed):
    from gated_delta_rule_kaczmarz_gb300.workloads import decode_inputs
    rng = np.random.default_rng(seed)
    d, dtype = [(64, "fp32"), (128, "bf16"), (128, "fp32"), (64, "bf16")][seed % 4]
    B, H, steps = int(rng.integers(1, 40)), int(rng.integers(1, 9)), int(rng.integers(1, 6))
    inp = decode_inputs(B, H, d, d, steps=steps, dtype=dtype, seed=seed)
    S = inp["S"].cuda()
    S_ref = inp["S"].double().numpy()
    tol = TOL[inp["q"].dtype]
    for t in range(steps):
        g = {n: inp[n][t].cuda() for n in ("q", "k", "v", "alpha", "eta")}
        o = kla.kla_decode_step(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], S)
        o_ref, S_ref = oracle.decode(inp["q"][t], inp["k"][t], inp["v"][t], inp["alpha"][t],
                                     inp["eta"][t], inp["eps"], S_ref)
        torch.cuda.synchronize()
        assert rel_err(o, o_ref) <= tol
    assert rel_err(S, S_ref) <= tol


@pytest.mark.parametrize("seed", [71, 72])
def test_random_noalloc(seed):
    """The no-allocation entry point gives the same results as kla_chunk_fwd
    and an OK device status."""
    rng = np.random.default_rng(seed)
    B, T, H = int(rng.integers(1, 4)), int(rng.integers(1, 400)), int(rng.integers(1, 4))
    inp = prefill_inputs(B, T, H, 128, 128, "bf16", seed=seed, s0_var=0.01)
    g = cuda(inp)
    o1, S1 = kla.kla_chunk_fwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"])
    o2, S2 = torch.empty_like(o1), torch.empty_like(S1)   # the entry point allocates nothing
    kla.kla_chunk_fwd_noalloc(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"],
                              o=o2, S_T=S2)
    assert kla.kla_chunk_fwd_noalloc_status() == binding.KLA_OK
    torch.testing.assert_close(o2, o1, rtol=0, atol=0)
    torch.testing.assert_close(S2, S1, rtol=0, atol=0)


# The launch-form boundaries on this GPU (152 SMs): the fused launch needs an
# even number of chunks and 2 B H <= 76; the two-launch state pass turns wide
# when 2 B H > 152.  Lengths on both sides of chunk (64-token) boundaries.
BOUNDARY = [(B, T, H) for (B, H) in ((19, 2), (13, 3), (38, 2), (39, 2))
            for T in (64, 65, 128, 129, 192, 193)]


@pytest.mark.parametrize("B,T,H", BOUNDARY)
def test_launch_form_boundaries(B, T, H):
    inp = prefill_inputs(B, T, H, 128, 128, "bf16", seed=B * 1000 + T + H, s0_var=0.01)
    g = cuda(inp)
    ws = torch.empty(kla.kla_chunk_fwd_workspace_size(B, T, H, 128, 128), dtype=torch.uint8,
                     device="cuda")
    o, S = kla.kla_chunk_fwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], inp["eps"], g["S0"],
                             workspace=ws)
    assert kla.kla_workspace_status(ws) == binding.KLA_OK
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                  inp["eps"], inp["S0"], nthreads=16)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2
