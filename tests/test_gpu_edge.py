"""GPU parity at the method's edge values, element by element against the fp64
oracle, on every path: the bf16 tensor-core kernels (single fused launch and
two launches), the fp32 CUDA-core kernel and the decode step.

  * a key of zero with eps = 0, where beta = eta / 0 is taken as 0 (the limit
    of the write term beta k e^T);
  * eta = 1, eps = 0: each write is the orthogonal projection onto
    {S : S^T k_t = v_t} (Kaczmarz Linear Attention summary, "Derivacao
    Teorica" and "Propriedades Chave" item 1), checked on the fp32 decode
    step and the fp32 prefill as S_t^T k_t = v_t;
  * alpha = 1e-30 on some tokens, several in one chunk, so that in-chunk
    decay products exp(g_t - g_s) fall below the fp32 range (the kernels form
    them from differences of cumulative logs and must produce 0, not NaN);
  * orthogonal keys k_t = c_t e_{i_t}, alpha = 1, eta = 1, eps = 0: write t
    overwrites row i_t of the state with v_t / c_t and leaves the others.

Tolerance: max|gpu - oracle| / max|oracle| per output tensor, 1e-4 for fp32
inputs and 2e-2 for bf16 inputs with the fp32 state."""
import numpy as np
import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300.workloads import decode_inputs, prefill_inputs
from tests._util import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu

# (name, B, T, H, d, dtype, launches per call): the single fused tensor-core
# launch needs an even number of chunks per sequence; three chunks take the
# two-launch path; fp32 takes the CUDA-core kernel.
PATHS = [
    ("tc_fused", 2, 256, 2, 128, "bf16", 1),
    ("tc_two_launch", 1, 192, 2, 128, "bf16", 2),
    ("fp32", 1, 200, 2, 64, "fp32", 1),
]


def _prefill(inp, launches=None, alpha_none=False):
    d = cuda(inp)
    n0 = kla.kla_launch_count()
    o, S = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], None if alpha_none else d["alpha"],
                             d["eta"], d["eps"], d["S0"])
    torch.cuda.synchronize()
    if launches is not None:
        assert kla.kla_launch_count() - n0 == launches
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"],
                                  None if alpha_none else inp["alpha"], inp["eta"], inp["eps"],
                                  inp["S0"], nthreads=8)
    return o, S, o_ref, S_ref


@pytest.mark.parametrize("name,B,T,H,d,dtype,launches", PATHS)
def test_zero_keys_with_eps_zero(name, B, T, H, d, dtype, launches):
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=300, s0_var=0.01, eps=0.0)
    # a few zero keys inside chunks (including a chunk's first and last row)
    for t in (0, 5, 6, 63, 64, 100, T - 1):
        inp["k"][:, t] = 0
    o, S, o_ref, S_ref = _prefill(inp, launches)
    tol = TOL[inp["q"].dtype]
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all()
    assert rel_err(o, o_ref) <= tol
    assert rel_err(S, S_ref) <= tol


@pytest.mark.parametrize("name,B,T,H,d,dtype,launches", PATHS)
def test_exact_projection_eta_one_eps_zero(name, B, T, H, d, dtype, launches):
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=301, s0_var=0.01, eps=0.0)
    inp["eta"].fill_(1.0)
    o, S, o_ref, S_ref = _prefill(inp, launches)
    tol = TOL[inp["q"].dtype]
    assert rel_err(o, o_ref) <= tol
    assert rel_err(S, S_ref) <= tol
    if dtype == "fp32":
        # the last write is a projection: S_T^T k_T = v_T (fp32 arithmetic)
        k = inp["k"][:, -1].double()                      # [B, H, d]
        v = inp["v"][:, -1].double()
        Sk = torch.einsum("bhij,bhi->bhj", S.cpu().double(), k)
        assert float((Sk - v).abs().max() / v.abs().max()) <= 1e-4


@pytest.mark.parametrize("dtype,d", [("fp32", 128), ("fp32", 64), ("bf16", 128)])
def test_decode_exact_projection_eta_one_eps_zero(dtype, d):
    """One decode step with eta = 1, eps = 0 leaves S_t^T k_t = v_t to fp32
    rounding (k and v are the stored values; the state and arithmetic are fp32)."""
    dec = decode_inputs(8, 4, d, d, steps=3, dtype=dtype, seed=302, eps=0.0)
    S = dec["S"].cuda()
    S_ref = dec["S"].double().numpy()
    for t in range(3):
        eta = torch.ones_like(dec["eta"][t])
        o = kla.kla_decode_step(dec["q"][t].cuda(), dec["k"][t].cuda(), dec["v"][t].cuda(),
                                dec["alpha"][t].cuda(), eta.cuda(), 0.0, S)
        torch.cuda.synchronize()
        o_ref, S_ref = oracle.decode(dec["q"][t], dec["k"][t], dec["v"][t], dec["alpha"][t], eta,
                                     0.0, S_ref)
        tol = TOL[dec["q"].dtype]
        assert rel_err(o, o_ref) <= tol and rel_err(S, S_ref) <= 1e-4
        k = dec["k"][t].double()
        v = dec["v"][t].double()
        Sk = torch.einsum("bhij,bhi->bhj", S.cpu().double(), k)
        assert float((Sk - v).abs().max() / v.abs().max()) <= 1e-4


@pytest.mark.parametrize("dtype,d", [("fp32", 64), ("bf16", 128)])
def test_decode_zero_key_eps_zero_and_tiny_alpha(dtype, d):
    dec = decode_inputs(8, 4, d, d, steps=2, dtype=dtype, seed=303, eps=0.0)
    dec["k"][0, :3] = 0            # zero keys: no write
    dec["alpha"][1, 2:5] = 1e-30   # the state decays to (almost) nothing
    S = dec["S"].cuda()
    S_ref = dec["S"].double().numpy()
    for t in range(2):
        o = kla.kla_decode_step(dec["q"][t].cuda(), dec["k"][t].cuda(), dec["v"][t].cuda(),
                                dec["alpha"][t].cuda(), dec["eta"][t].cuda(), 0.0, S)
        torch.cuda.synchronize()
        o_ref, S_ref = oracle.decode(dec["q"][t], dec["k"][t], dec["v"][t], dec["alpha"][t],
                                     dec["eta"][t], 0.0, S_ref)
        tol = TOL[dec["q"].dtype]
        assert torch.isfinite(S).all()
        assert rel_err(o, o_ref) <= tol and rel_err(S, S_ref) <= 1e-4


@pytest.mark.parametrize("name,B,T,H,d,dtype,launches", PATHS)
def test_tiny_alpha_underflows_in_chunk_decay(name, B, T, H, d, dtype, launches):
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=304, s0_var=0.01)
    # three consecutive tokens of 1e-30 inside chunk 0 (cumulative log decay
    # -207: exp underflows in fp32), one at a chunk's first row, one at a
    # chunk's last row, and one in a later chunk
    tiny = [3, 4, 5, 64, 127, 150]
    inp["alpha"][:, [t for t in tiny if t < T]] = 1e-30
    o, S, o_ref, S_ref = _prefill(inp, launches)
    tol = TOL[inp["q"].dtype]
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all()
    assert rel_err(o, o_ref) <= tol
    assert rel_err(S, S_ref) <= tol


def _orthogonal_inputs(B, T, H, d, dtype, seed):
    """k_t = c_t e_{i_t} with distinct i_t per (sequence, head), c_t a power of
    two (exact in bf16); alpha = 1, eta = 1, eps = 0."""
    assert T <= d
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=seed, s0_var=0.01, eps=0.0)
    rng = np.random.default_rng(seed)
    idx = np.stack([np.stack([rng.permutation(d)[:T] for _ in range(H)], 1) for _ in range(B)])
    c = 2.0 ** rng.integers(-1, 3, size=(B, T, H))
    k = np.zeros((B, T, H, d), np.float32)
    for b in range(B):
        for t in range(T):
            for h in range(H):
                k[b, t, h, idx[b, t, h]] = c[b, t, h]
    inp["k"] = torch.from_numpy(k).to(inp["q"].dtype)
    inp["alpha"].fill_(1.0)
    inp["eta"].fill_(1.0)
    return inp, idx, c


@pytest.mark.parametrize("name,B,T,H,d,dtype,launches", [
    ("tc_fused", 2, 128, 2, 128, "bf16", 1),
    ("tc_two_launch", 40, 128, 2, 128, "bf16", 2),     # 160 state CTAs: two launches
    ("fp32", 2, 64, 2, 64, "fp32", 1),
])
@pytest.mark.parametrize("alpha_none", [False, True])
def test_orthogonal_keys_overwrite_rows(name, B, T, H, d, dtype, launches, alpha_none):
    inp, idx, c = _orthogonal_inputs(B, T, H, d, dtype, seed=305)
    o, S, o_ref, S_ref = _prefill(inp, launches, alpha_none=alpha_none)
    tol = TOL[inp["q"].dtype]
    assert rel_err(o, o_ref) <= tol
    assert rel_err(S, S_ref) <= tol
    # the property itself: row i_t of S_T is v_t / c_t, untouched rows keep S0
    S_cpu = S.cpu().double()
    S0 = inp["S0"].double()
    v = inp["v"].double()
    expect = S0.clone()
    for b in range(B):
        for t in range(T):
            for h in range(H):
                expect[b, h, idx[b, t, h]] = v[b, t, h] / c[b, t, h]
    assert float((S_cpu - expect).abs().max() / expect.abs().max()) <= tol


def test_decode_orthogonal_keys_overwrite_rows():
    """Decode steps with orthogonal keys, alpha = 1, eta = 1, eps = 0 on the
    fp32 state: each step sets row i_t to v_t / c_t to fp32 rounding."""
    B, H, d, steps = 4, 2, 128, 6
    dec = decode_inputs(B, H, d, d, steps=steps, dtype="fp32", seed=306, eps=0.0)
    rng = np.random.default_rng(306)
    S = dec["S"].cuda()
    expect = dec["S"].double().clone()
    for t in range(steps):
        idx = rng.integers(0, d, size=(B, H))
        c = 2.0 ** rng.integers(-1, 3, size=(B, H))
        k = torch.zeros(B, H, d)
        for b in range(B):
            for h in range(H):
                k[b, h, idx[b, h]] = float(c[b, h])
                expect[b, h, idx[b, h]] = dec["v"][t, b, h].double() / c[b, h]
        one = torch.ones(B, H)
        kla.kla_decode_step(dec["q"][t].cuda(), k.cuda(), dec["v"][t].cuda(), one.cuda(),
                            one.cuda(), 0.0, S)
    torch.cuda.synchronize()
    assert float((S.cpu().double() - expect).abs().max() / expect.abs().max()) <= 1e-5
