"""kla_chunk_fwd_noalloc: the prefill entry point for callers that cannot
allocate device memory (a framework owning every device byte through its own
pool, a plugin interface handed only input and output pointers, a serving
loop that cannot pay cudaMalloc's device-wide synchronisation).  It runs the
same kernels as kla_chunk_fwd with the library's built-in device array as
workspace.  This file is collected last so that a failure here cannot hide
the other tests' results."""
import ctypes

import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
import oracle
from gated_delta_rule_kaczmarz_gb300 import binding
from gated_delta_rule_kaczmarz_gb300.workloads import prefill_inputs
from tests._util import TOL, rel_err

LIMIT = 64 * 1024 * 1024


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.gpu
def test_noalloc_matches_kla_chunk_fwd_two_calls_in_a_row():
    """Two differently shaped calls in a row share the built-in array (the
    second reuses what the first left in it): each matches kla_chunk_fwd with
    its own workspace, the device status of each is OK, and the smaller call
    is also checked against the fp64 oracle."""
    lib = binding.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed, (B, T, H) in ((70, (2, 300, 4)), (71, (4, 2048, 8))):
        inp = prefill_inputs(B, T, H, 128, 128, "bf16", seed=seed, s0_var=0.01)
        d = {n: (x.cuda() if isinstance(x, torch.Tensor) else x) for n, x in inp.items()}
        o_ref, S_ref = kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], d["eps"],
                                         d["S0"])
        o = torch.empty_like(o_ref)
        S_T = torch.empty_like(S_ref)
        st = lib.kla_chunk_fwd_noalloc(_ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]), _ptr(d["alpha"]),
                                       _ptr(d["eta"]), d["eps"], _ptr(d["S0"]), _ptr(o), _ptr(S_T),
                                       B, T, H, 128, 128, 64, binding.KLA_DTYPE_BF16, stream)
        assert st == binding.KLA_OK, lib.kla_last_error_message()
        assert lib.kla_chunk_fwd_noalloc_status(stream) == binding.KLA_OK, \
            lib.kla_last_error_message()
        torch.cuda.synchronize()
        tol = TOL[torch.bfloat16]
        assert rel_err(o, o_ref.cpu().double().numpy()) <= tol
        assert rel_err(S_T, S_ref.cpu().double().numpy()) <= tol
        if T <= 300:
            o_or, S_or = oracle.forward(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                        inp["eps"], inp["S0"], nthreads=8)
            assert rel_err(o, o_or) <= tol
            assert rel_err(S_T, S_or) <= tol


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_array():
    # 1 x 131072 tokens x 1 head needs about 84 MB of workspace (> 64 MiB);
    # the tensors are real so nothing could be read out of bounds even if the
    # size check were missing.
    B, T, H = 1, 131072, 1
    assert kla.kla_chunk_fwd_workspace_size(B, T, H, 128, 128) > LIMIT
    q = torch.zeros(B, T, H, 128, dtype=torch.bfloat16, device="cuda")
    a = torch.ones(B, T, H, device="cuda")
    with pytest.raises(kla.KlaError) as ei:
        kla.kla_chunk_fwd_noalloc(q, q, q, a, a, 1e-6)
    assert ei.value.status == binding.KLA_ERR_WORKSPACE
    assert "scratch" in str(ei.value)
