"""kla_chunk: the forward under torch.autograd, whose backward is
kla_chunk_bwd; gradients of a weighted sum of o and S_T against the backward
oracle (max|err| / max|oracle| <= 1e-4 fp32, 2e-2 bf16)."""
import numpy as np
import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300.workloads import prefill_inputs
from tests._util import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,T,H,d,dtype", [(1, 96, 2, 64, "fp32"), (2, 192, 2, 128, "bf16")])
def test_autograd_matches_oracle(B, T, H, d, dtype):
    inp = prefill_inputs(B, T, H, d, d, dtype, seed=500 + T, s0_var=0.01)
    rng = np.random.default_rng(501)
    w_o = torch.from_numpy(rng.standard_normal((B, T, H, d)).astype(np.float32)).to(inp["q"].dtype)
    w_S = torch.from_numpy((0.1 * rng.standard_normal((B, H, d, d))).astype(np.float32))
    leaves = {n: inp[n].cuda().requires_grad_(True) for n in ("q", "k", "v", "alpha", "eta", "S0")}
    o, S = kla.kla_chunk(leaves["q"], leaves["k"], leaves["v"], leaves["alpha"], leaves["eta"],
                         inp["eps"], leaves["S0"])
    loss = (o.float() * w_o.cuda().float()).sum() + (S * w_S.cuda()).sum()
    loss.backward()
    torch.cuda.synchronize()
    ref = oracle.backward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"], inp["eps"],
                          inp["S0"], w_o, w_S, nthreads=8)
    tol = TOL[inp["q"].dtype]
    for name, r in zip(("q", "k", "v", "alpha", "eta", "S0"), ref):
        assert rel_err(leaves[name].grad, r) <= tol, name
