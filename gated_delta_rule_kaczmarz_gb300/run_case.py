"""Runs one named workload through the public API a few times on cuda:0.

    python -m gated_delta_rule_kaczmarz_gb300.run_case layer_prefill --calls 3
    python -m gated_delta_rule_kaczmarz_gb300.run_case decode --B 128 --calls 3
    python -m gated_delta_rule_kaczmarz_gb300.run_case backward --calls 2

A fixed, short launch sequence for profilers: prefill and varlen workloads
run ``calls`` full calls (one chunkwise forward each); ``decode`` runs
``calls`` single-token steps on a [B, 16, 128, 128] state; ``ccq`` runs
the CCQ query contraction on the layer_prefill workload's q and k; ``backward``
runs the backward pass of the layer_prefill workload (d_o ~ N(0,1), dS_T ~
N(0,0.01)).  Inputs are
uploaded before the first call.  Prints one line with the mean time per call
(CUDA events, inputs resident; not a benchmark figure when run under a
profiler).
"""
from __future__ import annotations

import argparse
import sys

import torch

from . import binding as kla
from .workloads import WORKLOADS, decode_inputs


def _dev(inp):
    return {n: (x.cuda() if isinstance(x, torch.Tensor) else x) for n, x in inp.items()}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(list(WORKLOADS) + ["decode", "ccq", "backward"]))
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--B", type=int, default=128, help="batch of the decode case")
    a = ap.parse_args(argv)
    calls = []
    if a.case == "backward":
        wl = WORKLOADS["layer_prefill"]
        inp = _dev(wl.make())
        gen = torch.Generator(device="cuda").manual_seed(11)
        do = torch.randn((wl.B, wl.T, wl.H, wl.d), device="cuda", generator=gen).to(torch.bfloat16)
        dST = 0.1 * torch.randn((wl.B, wl.H, wl.d, wl.d), device="cuda", generator=gen)
        ws = torch.empty(kla.kla_chunk_bwd_workspace_size(wl.B, wl.T, wl.H, wl.d),
                         dtype=torch.uint8, device="cuda")
        calls = [lambda: kla.kla_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                           wl.eps, inp["S0"], do, dST, workspace=ws)] * a.calls
    elif a.case == "ccq":
        # the CCQ query contraction on the layer workload's q and k
        inp = _dev(WORKLOADS["layer_prefill"].make())
        lam = torch.full(inp["eta"].shape, 0.5, dtype=torch.float32, device="cuda")
        calls = [lambda: kla.kla_ccq_query(inp["q"], inp["k"], lam)] * a.calls
    elif a.case == "decode":
        inp = _dev(decode_inputs(a.B, 16, 128, 128, steps=a.calls, dtype="bf16", seed=3))
        S = inp["S"]
        o = torch.empty_like(inp["v"][0])
        for t in range(a.calls):
            calls.append(lambda t=t: kla.kla_decode_step(
                inp["q"][t], inp["k"][t], inp["v"][t], inp["alpha"][t], inp["eta"][t],
                inp["eps"], S, o=o))
    else:
        wl = WORKLOADS[a.case]
        inp = _dev(wl.make())
        if wl.kind == "varlen":
            f = lambda: kla.kla_chunk_fwd_varlen(inp["q"], inp["k"], inp["v"], inp["alpha"],
                                                 inp["eta"], inp["eps"], inp["cu_seqlens"],
                                                 inp["S0"])
        else:
            f = lambda: kla.kla_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["alpha"],
                                          inp["eta"], inp["eps"], inp["S0"])
        calls = [f] * a.calls
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for c in calls:
        c()
    e1.record()
    torch.cuda.synchronize()
    print(f"{a.case}: {len(calls)} calls, {e0.elapsed_time(e1) * 1e3 / max(1, len(calls)):.1f} us/call")
    return 0


if __name__ == "__main__":
    sys.exit(main())
