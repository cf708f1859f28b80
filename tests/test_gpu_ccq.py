"""GPU parity of the CCQ query contraction (kla_ccq_query, kla_ccq_query_step)
and of a whole CCQ layer (the KLA forward on q_clean) against the fp64
oracle; error measure max|gpu - oracle| / max|oracle|, 1e-4 (fp32) and 2e-2
(bf16)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300.workloads import prefill_inputs
from tests._util import TOL, cuda, rel_err

pytestmark = pytest.mark.gpu


def _lam(shape, seed):
    rng = np.random.default_rng(seed)
    return torch.from_numpy((1.0 / (1.0 + np.exp(-rng.standard_normal(shape)))).astype(np.float32))


def _stats(B, H, d, seed):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((B, H, 50, d)) / np.sqrt(d)
    Ms = np.einsum("bhti,bhtj->bhij", K, K).astype(np.float32)
    ms = K.sum(2).astype(np.float32)
    ns = np.full((B, H), 50.0, np.float32)
    return tuple(torch.from_numpy(x) for x in (Ms, ms, ns))


@pytest.mark.parametrize("B,T,H,d,dtype,with_stats", [
    (2, 200, 2, 64, "fp32", False), (1, 130, 2, 128, "fp32", True),
    (2, 257, 2, 128, "bf16", False), (1, 64, 3, 128, "bf16", True), (2, 1, 2, 64, "bf16", True),
    # tensor-core path: whole and ragged 128-token blocks, several segments
    # per sequence, sequences shorter than a block
    (2, 256, 2, 128, "bf16", True), (3, 448, 2, 128, "bf16", False), (1, 323, 5, 128, "bf16", True),
    (80, 1, 1, 128, "bf16", True), (3, 40, 2, 128, "bf16", False)])
def test_ccq_query_parity(B, T, H, d, dtype, with_stats):
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=120 + T)
    lam = _lam((B, T, H), 7)
    st0 = _stats(B, H, d, 8) if with_stats else None
    g = cuda(inp)
    qc, (Ms, ms, ns) = kla.kla_ccq_query(g["q"], g["k"], lam.cuda(),
                                         None if st0 is None else tuple(x.cuda() for x in st0))
    torch.cuda.synchronize()
    qc_ref, (Ms_ref, ms_ref, ns_ref) = oracle.ccq_query(inp["q"], inp["k"], lam, st0)
    tol = TOL[inp["q"].dtype]
    assert rel_err(qc, qc_ref) <= tol
    assert rel_err(Ms, Ms_ref) <= 1e-5 and rel_err(ms, ms_ref) <= 1e-5
    assert np.array_equal(ns.cpu().numpy(), ns_ref)


def test_ccq_layer_end_to_end():
    """A CCQ-KLA layer: q_clean on the GPU, then the tensor-core forward on it,
    against the oracle's q_clean and forward."""
    inp = prefill_inputs(2, 256, 2, 128, 128, "bf16", seed=130, s0_var=0.01)
    lam = _lam((2, 256, 2), 9)
    g = cuda(inp)
    qc, _ = kla.kla_ccq_query(g["q"], g["k"], lam.cuda())
    o, S = kla.kla_chunk_fwd(qc, g["k"], g["v"], g["alpha"], g["eta"], g["eps"], g["S0"])
    torch.cuda.synchronize()
    qc_ref, _ = oracle.ccq_query(inp["q"], inp["k"], lam)
    o_ref, S_ref = oracle.forward(qc_ref, inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                  inp["eps"], inp["S0"], nthreads=8)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2


@pytest.mark.parametrize("d,dtype", [(64, "fp32"), (128, "bf16")])
def test_ccq_step_equals_prefill(d, dtype):
    """Token-by-token CCQ steps from given statistics equal the chunked pass."""
    B, T, H = 2, 9, 3
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=140 + d)
    lam = _lam((B, T, H), 10)
    st0 = _stats(B, H, d, 11)
    g = cuda(inp)
    Ms, ms, ns = (x.cuda().clone() for x in st0)
    outs = []
    for t in range(T):
        outs.append(kla.kla_ccq_query_step(g["q"][:, t].contiguous(), g["k"][:, t].contiguous(),
                                           lam[:, t].contiguous().cuda(), Ms, ms, ns))
    torch.cuda.synchronize()
    qc_ref, (Ms_ref, ms_ref, ns_ref) = oracle.ccq_query(inp["q"], inp["k"], lam, st0)
    tol = TOL[inp["q"].dtype]
    assert rel_err(torch.stack(outs, 1), qc_ref) <= tol
    assert rel_err(Ms, Ms_ref) <= 1e-5
    assert np.array_equal(ns.cpu().numpy(), ns_ref)


@pytest.mark.parametrize("B,T,H", [(2, 256, 2), (2, 320, 2), (40, 256, 4), (1, 2048, 2)])
def test_ccq_tensor_core_launches(B, T, H):
    """bf16 dk 128 streams 128-token blocks through the tensor cores in one
    launch: with few (sequence, head) pairs each sequence is cut into segments
    whose CTAs first add the K^T K of the blocks before them; the status word
    in the workspace stays 0 and the statistics are exact."""
    d = 128
    inp = prefill_inputs(B, T, H, d, d, "bf16", seed=150)
    lam = _lam((B, T, H), 12)
    st0 = _stats(B, H, d, 15)
    g = cuda(inp)
    ws = torch.zeros(kla.kla_ccq_query_workspace_size(B, T, H, d), dtype=torch.uint8,
                     device="cuda")
    stats = tuple(x.cuda() for x in st0)
    kla.kla_ccq_query(g["q"], g["k"], lam.cuda(), stats, workspace=ws)   # sets attributes
    torch.cuda.synchronize()
    n0 = kla.kla_launch_count()
    qc, (Ms, ms, ns) = kla.kla_ccq_query(g["q"], g["k"], lam.cuda(), stats, workspace=ws)
    torch.cuda.synchronize()
    assert kla.kla_launch_count() - n0 == 1
    assert kla.kla_workspace_status(ws) == 0
    qc_ref, (Ms_ref, ms_ref, ns_ref) = oracle.ccq_query(inp["q"], inp["k"], lam, st0)
    assert rel_err(qc, qc_ref) <= TOL[inp["q"].dtype]
    assert rel_err(Ms, Ms_ref) <= 1e-5 and rel_err(ms, ms_ref) <= 1e-5
    assert np.array_equal(ns.cpu().numpy(), ns_ref)


def test_ccq_full_size_sampled():
    """The layer workload (B4 H8 T2048 d128 bf16): q_clean and the final
    statistics of two sampled (sequence, head) units against the oracle run on
    those units alone."""
    from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS
    wl = WORKLOADS["layer_prefill"]
    inp = wl.make()
    lam = _lam((wl.B, wl.T, wl.H), 13)
    g = cuda(inp)
    qc, (Ms, ms, ns) = kla.kla_ccq_query(g["q"], g["k"], lam.cuda())
    torch.cuda.synchronize()
    for b, h in ((0, 0), (3, 5)):
        q1 = inp["q"][b:b + 1, :, h:h + 1].contiguous()
        k1 = inp["k"][b:b + 1, :, h:h + 1].contiguous()
        l1 = lam[b:b + 1, :, h:h + 1].contiguous()
        ref, (M_ref, m_ref, n_ref) = oracle.ccq_query(q1, k1, l1)
        assert rel_err(qc[b:b + 1, :, h:h + 1], ref) <= TOL[inp["q"].dtype]
        assert rel_err(Ms[b:b + 1, h:h + 1], M_ref) <= 1e-5
        assert rel_err(ms[b:b + 1, h:h + 1], m_ref) <= 1e-5
        assert float(ns[b, h]) == float(n_ref.reshape(-1)[0])


def test_ccq_stats_carry_on_tensor_cores():
    """Two tensor-core calls with the statistics carried equal one call over
    the concatenation (bf16 d 128)."""
    B, H, d = 2, 2, 128
    inp = prefill_inputs(B, 512, H, d, d, "bf16", seed=170)
    lam = _lam((B, 512, H), 14).cuda()
    g = cuda(inp)
    qc, st = kla.kla_ccq_query(g["q"], g["k"], lam)
    qa, sa = kla.kla_ccq_query(g["q"][:, :256].contiguous(), g["k"][:, :256].contiguous(),
                               lam[:, :256].contiguous())
    qb, sb = kla.kla_ccq_query(g["q"][:, 256:].contiguous(), g["k"][:, 256:].contiguous(),
                               lam[:, 256:].contiguous(), sa)
    torch.cuda.synchronize()
    ref = qc.double().cpu().numpy()
    assert rel_err(torch.cat([qa, qb], 1), ref) <= 2e-2
    for x, y in zip(sb, st):
        assert rel_err(x, y.double().cpu().numpy()) <= 1e-5


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "fp32")])
def test_ccq_lambda_zero_is_identity(d, dtype):
    """lambda = 0 leaves the query unchanged (CCQ, "O Mecanismo": q_clean =
    (I - lambda Sigma) q), bit for bit, on the tensor-core and CUDA-core
    paths, while the statistics still advance."""
    B, T, H = 2, 300, 2
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=180)
    lam = torch.zeros(B, T, H)
    g = cuda(inp)
    qc, (Ms, ms, ns) = kla.kla_ccq_query(g["q"], g["k"], lam.cuda())
    torch.cuda.synchronize()
    assert torch.equal(qc.cpu(), inp["q"])
    _, (Ms_ref, ms_ref, ns_ref) = oracle.ccq_query(inp["q"], inp["k"], lam)
    assert rel_err(Ms, Ms_ref) <= 1e-5 and rel_err(ms, ms_ref) <= 1e-5


def test_ccq_keys_with_a_common_mean_and_zero_keys():
    """Keys k_t = mu + noise with |mu| of the order of the noise's norm (the
    covariance is then a small difference M/n - mu mu^T), a few zero keys
    (they still count in n_t), over several segments per sequence."""
    B, T, H, d = 1, 1000, 2, 128
    inp = prefill_inputs(B, T, H, d, d, "bf16", seed=181)
    rng = np.random.default_rng(182)
    mu = rng.standard_normal((1, 1, H, d)) / np.sqrt(d)
    k = inp["k"].double().numpy() * 0.5 + mu
    k[:, [0, 7, 300, 999]] = 0.0
    inp["k"] = torch.from_numpy(k).to(torch.bfloat16)
    lam = _lam((B, T, H), 183)
    g = cuda(inp)
    qc, (Ms, ms, ns) = kla.kla_ccq_query(g["q"], g["k"], lam.cuda())
    torch.cuda.synchronize()
    qc_ref, (Ms_ref, ms_ref, ns_ref) = oracle.ccq_query(inp["q"], inp["k"], lam)
    assert rel_err(qc, qc_ref) <= TOL[inp["q"].dtype]
    assert rel_err(Ms, Ms_ref) <= 1e-5 and rel_err(ms, ms_ref) <= 1e-5
    assert np.array_equal(ns.cpu().numpy(), ns_ref)
