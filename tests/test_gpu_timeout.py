"""The timeout path of the bounded device waits, made to run on the GPU
without a hang or a fault.

The single-launch prefill's state pass waits for each chunk pair to be
published by the phase-1 workers of the same launch; every such wait is
bounded.  The test hook KLA_TEST_FLAG_WAIT=<cycles> sets that bound for one
call and makes the state pass first wait on a header word of the workspace
that nothing sets.  With a bound of 0 the wait runs out at once: the call must
record KLA_ERR_TIMEOUT in the workspace status, its other warps must leave
without sitting out their own (one-second) bounds, and the next normal call on
the same workspace must be exact again."""
import time

import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300 import binding
from gated_delta_rule_kaczmarz_gb300.workloads import prefill_inputs
from tests._util import cuda, rel_err

pytestmark = pytest.mark.gpu


def _call(d, ws):
    n0 = kla.kla_launch_count()
    o, S = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"], d["S0"],
                             workspace=ws)
    return o, S, kla.kla_launch_count() - n0


@pytest.mark.parametrize("B,T,H", [(2, 256, 2), (4, 1024, 2)])
def test_flag_wait_that_runs_out_reports_timeout(monkeypatch, B, T, H):
    inp = prefill_inputs(B, T, H, 128, 128, "bf16", seed=400 + T, s0_var=0.01)
    d = cuda(inp)
    ws = torch.empty(kla.kla_chunk_fwd_workspace_size(B, T, H, 128, 128), dtype=torch.uint8,
                     device="cuda")
    _call(d, ws)                                   # warm-up: context, attributes
    assert kla.kla_workspace_status(ws) == binding.KLA_OK

    monkeypatch.setenv("KLA_TEST_FLAG_WAIT", "0")
    t0 = time.perf_counter()
    _, _, launches = _call(d, ws)
    with pytest.raises(kla.KlaError) as ei:
        kla.kla_workspace_status(ws)               # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert launches == 1                           # the single fused launch ran
    assert ei.value.status == binding.KLA_ERR_TIMEOUT
    # sibling warps stopped waiting as soon as the wait ran out (each of their
    # own bounds is about one second of SM clock)
    assert elapsed < 0.5, elapsed
    torch.cuda.synchronize()                       # the context is still usable

    monkeypatch.delenv("KLA_TEST_FLAG_WAIT")
    o, S, launches = _call(d, ws)
    assert kla.kla_workspace_status(ws) == binding.KLA_OK
    assert launches == 1
    o_ref, S_ref = oracle.forward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                  inp["eps"], inp["S0"], nthreads=8)
    assert rel_err(o, o_ref) <= 2e-2
    assert rel_err(S, S_ref) <= 2e-2
