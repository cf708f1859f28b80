#!/usr/bin/env python
"""Benchmark of the KLA hot path on one GB300 (or N independent replicas).

Step = one chunkwise prefill (kla_chunk_fwd) of the 0.4B-scale layer
workload: B=4, H=8, T=2048, dk=dv=128, chunk 64, bf16 q/k/v, fp32
alpha/eta/state, S0 ~ N(0,0.01), returning o and S_T.  The same run times
the batched decode workload (B=256, H=16, d=128, 64 in-place steps) and
reports it under "decode".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: CUDA events on the launching stream around each step; L2 is flushed
(256 MiB write) between timed prefill steps, outside the events; the decode
state (268 MB) is larger than L2.  The end-to-end figure copies every step's
inputs from pinned host memory and its outputs back, pipelined over two
device buffer sets (copies in, compute and copies out of consecutive steps
overlap on three streams); it is the total time of all steps / steps.  For N > 1 (torchrun) every rank runs its
own replica; times are max-reduced over ranks and value = total tokens / time.
The reference arm (--impl reference) times the fp64 CPU oracle on the host.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KLA chunkwise prefill tokens/s & % roofline; decode steps/s at B=256"
# DRAM bytes (read + write) of one prefill launch (fused_kernel), one decode
# launch scaled to B=256 and one CCQ query call (its two launches), from the ncu
# captures summarised in profiles/ (fused_kernel_layer_prefill.md,
# decode_kernel_b128.md, ccq_layer_prefill.md).
TRAFFIC_PREFILL = 68.26e6
TRAFFIC_CCQ = 48.5e6 + 51.6e6
TRAFFIC_DECODE = 2 * (135.83e6 + 74.59e6)
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
BYTES_PER_TOKEN_HEAD = 1032          # q,k,v,o bf16 (4 x 256 B) + alpha, eta fp32 (8 B)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""
    QUERY = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 10]
        mine = [r for r in rows if self.bus_id and self.bus_id.endswith(r[1].strip().lower()[-12:])]
        if not mine and rows:
            idx = rows[0][0]
            mine = [r for r in rows if r[0] == idx]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in mine:
            try:
                sm.append(float(r[2]))
                smax.append(float(r[3]))
            except ValueError:
                continue
            for n, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- CPU oracle legs
def oracle_sample(inp, heads, tokens, nthreads):
    """Runs the fp64 oracle on `heads` (b, h) units of the first `tokens`
    tokens; returns (seconds, token-heads processed)."""
    import oracle
    B, T, H, _ = inp["q"].shape
    units = [(u // H, u % H) for u in range(B * H)][:heads]
    sel = lambda x: x[[b for b, _ in units], :tokens, [h for _, h in units]][:, :, None]
    args = [sel(inp[n]).contiguous() for n in ("q", "k", "v", "alpha", "eta")]
    S0 = None if inp["S0"] is None else inp["S0"][[b for b, _ in units], [h for _, h in units]][:, None]
    # convert before timing (the oracle's input is fp64)
    import numpy as np
    conv = [np.ascontiguousarray(a.double().numpy()) for a in args]
    S0c = None if S0 is None else np.ascontiguousarray(S0.double().numpy())
    t0 = time.perf_counter()
    oracle.forward(*conv[:5], inp["eps"], S0c, nthreads=nthreads)
    return time.perf_counter() - t0, len(units) * tokens


def reference_arm(args):
    """--impl reference: the fp64 CPU oracle, as it stands, on the host cores.
    Each step is a bounded sample of the layer workload: one (b, h) unit per
    core (at most 32), 512 tokens each."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS
    wl = WORKLOADS["layer_prefill"]
    inp = wl.make()
    cores = os.cpu_count() or 1
    heads = min(cores, wl.B * wl.H)
    tokens = 512
    for _ in range(args.warmup):
        oracle_sample(inp, heads, tokens, cores)
    total, work = 0.0, 0
    for _ in range(args.steps):
        s, w = oracle_sample(inp, heads, tokens, cores)
        total += s
        work += w
    value = (work / wl.H) / total
    sample = f"{heads} (b,h) units x {tokens} tokens of the layer workload per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "layer_prefill", "B": wl.B, "T": wl.T, "H": wl.H, "dk": wl.d,
                   "dv": wl.d, "chunk": wl.chunk, "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------- our arm
def time_prefill(args, world, dev):
    import torch

    import gated_delta_rule_kaczmarz_gb300 as kla
    from gated_delta_rule_kaczmarz_gb300 import binding
    from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS

    wl = WORKLOADS["layer_prefill"]
    inp_cpu = wl.make()
    B, T, H, d = wl.B, wl.T, wl.H, wl.d
    g = {n: (x.to(dev) if isinstance(x, torch.Tensor) else x) for n, x in inp_cpu.items()}
    o = torch.empty((B, T, H, d), dtype=torch.bfloat16, device=dev)
    S_T = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    wsb = kla.kla_chunk_fwd_workspace_size(B, T, H, d, d, 64, binding.KLA_DTYPE_BF16)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call(q, k, v, a, e, s0, out, st):
        kla.kla_chunk_fwd(q, k, v, a, e, wl.eps, s0, o=out, S_T=st, workspace=ws, stream=stream)

    def step():
        call(g["q"], g["k"], g["v"], g["alpha"], g["eta"], g["S0"], o, S_T)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    sampler = ClockSampler(bus).start()
    time.sleep(0.3)
    n0 = kla.kla_launch_count()
    evs = []
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    launches = kla.kla_launch_count() - n0
    times = [a.elapsed_time(b) for a, b in evs]
    barrier(world)

    # end to end through the public API from pinned host buffers: every step
    # copies its own inputs (q, k, v, alpha, eta, S0) in and its outputs (o,
    # S_T) out.  Steps are pipelined over two device buffer sets: step i+1's
    # inputs and step i-1's outputs move on their own streams while step i
    # computes (the L2 flush stays on the compute stream before every step).
    host = {n: (x.pin_memory() if isinstance(x, torch.Tensor) else x) for n, x in inp_cpu.items()}
    names = ("q", "k", "v", "alpha", "eta", "S0")
    nb = 2
    dbuf = [{n: torch.empty_like(g[n]) for n in names} for _ in range(nb)]
    obuf = [(torch.empty_like(o), torch.empty_like(S_T)) for _ in range(nb)]
    hout = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(),
             torch.empty(S_T.shape, dtype=S_T.dtype).pin_memory()) for _ in range(nb)]
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = o.numel() * o.element_size() + S_T.numel() * S_T.element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(nb)]
    ev_done = [torch.cuda.Event() for _ in range(nb)]
    ev_out = [torch.cuda.Event() for _ in range(nb)]
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(s_in)
    stream.wait_event(t_start)
    s_out.wait_event(t_start)
    for i in range(args.steps):
        bi = i % nb
        if i >= nb:
            s_in.wait_event(ev_done[bi])          # step i-2 finished reading these inputs
        with torch.cuda.stream(s_in):
            for n in names:
                dbuf[bi][n].copy_(host[n], non_blocking=True)
            ev_in[bi].record(s_in)
        stream.wait_event(ev_in[bi])
        if i >= nb:
            stream.wait_event(ev_out[bi])         # step i-2's outputs have left
        flush.zero_()
        d = dbuf[bi]
        kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], wl.eps, d["S0"],
                          o=obuf[bi][0], S_T=obuf[bi][1], workspace=ws, stream=stream)
        ev_done[bi].record(stream)
        s_out.wait_event(ev_done[bi])
        with torch.cuda.stream(s_out):
            hout[bi][0].copy_(obuf[bi][0], non_blocking=True)
            hout[bi][1].copy_(obuf[bi][1], non_blocking=True)
            ev_out[bi].record(s_out)
    s_out.wait_stream(stream)
    s_out.wait_stream(s_in)
    t_end.record(s_out)
    torch.cuda.synchronize()
    e2e_total_ms = t_start.elapsed_time(t_end)
    e2e_times = [e2e_total_ms / args.steps] * args.steps
    clocks = sampler.stop()
    return dict(wl=wl, times=times, e2e_times=e2e_times, h2d=h2d, d2h=d2h, launches=launches,
                clocks=clocks, inp_cpu=inp_cpu, kernels_per_call=launches / max(1, args.steps))


def time_decode(args, dev, reps):
    import torch

    import gated_delta_rule_kaczmarz_gb300 as kla
    from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS

    wl = WORKLOADS["decode_b256"]
    inp = wl.make()
    S = inp["S"].to(dev)
    per = {n: inp[n].to(dev) for n in ("q", "k", "v", "alpha", "eta")}
    steps = per["q"].shape[0]
    o = torch.empty((wl.B, wl.H, wl.d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def run():
        for t in range(steps):
            kla.kla_decode_step(per["q"][t], per["k"][t], per["v"][t], per["alpha"][t],
                                per["eta"][t], wl.eps, S, o=o, stream=stream)

    run()
    torch.cuda.synchronize()
    evs = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = sum(ms)
    n_launch = reps * steps
    BH = wl.B * wl.H
    bytes_per_launch = BH * (2 * wl.d * wl.d * 4 + 4 * wl.d * 2 + 8)
    avg_launch_s = total_ms / 1e3 / n_launch
    return dict(wl=wl, steps_per_s=n_launch / (total_ms / 1e3), avg_launch_s=avg_launch_s,
                bytes_per_launch=bytes_per_launch)


def time_ccq(args, dev, reps):
    """CCQ read-side contraction on the layer workload (bf16, B4 H8 T2048
    d128, lambda ~ sigmoid(N(0,1))): kla_ccq_query alone, and a whole CCQ
    layer (kla_ccq_query then kla_chunk_fwd on q_clean).  Inputs resident, L2
    flushed between timed calls."""
    import numpy as np
    import torch

    import gated_delta_rule_kaczmarz_gb300 as kla
    from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS

    wl = WORKLOADS["layer_prefill"]
    inp = wl.make()
    g = {n: (x.to(dev) if isinstance(x, torch.Tensor) else x) for n, x in inp.items()}
    rng = np.random.default_rng(5)
    lam = torch.from_numpy((1.0 / (1.0 + np.exp(-rng.standard_normal((wl.B, wl.T, wl.H)))))
                           .astype(np.float32)).to(dev)
    qc = torch.empty_like(g["q"])
    ws = torch.empty(max(1, kla.kla_ccq_query_workspace_size(wl.B, wl.T, wl.H, wl.d)),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def query():
        kla.kla_ccq_query(g["q"], g["k"], lam, q_clean=qc, return_stats=False, workspace=ws,
                          stream=stream)

    def layer():
        query()
        kla.kla_chunk_fwd(qc, g["k"], g["v"], g["alpha"], g["eta"], wl.eps, g["S0"],
                          stream=stream)

    out = {}
    for name, f in (("query", query), ("layer", layer)):
        for _ in range(2):
            f()
        torch.cuda.synchronize()
        ms = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            f()
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        out[name] = sum(ms) / len(ms)
    th = wl.B * wl.T * wl.H
    # algorithmic bytes of the query: q and k read, q_clean written (bf16), lambda read
    nbytes = th * (3 * wl.d * 2 + 4)
    return dict(wl=wl, query_ms=out["query"], layer_ms=out["layer"], bytes=nbytes)


def time_bwd(args, dev, reps):
    """Backward pass (kla_chunk_bwd) on the layer workload (bf16, B4 H8 T2048
    d128): the gradients of sum <d_o, o> + <dS_T, S_T> with d_o ~ N(0,1) and
    dS_T ~ N(0, 0.01).  Inputs and workspace resident, L2 flushed between
    timed calls; also each of the three kernels alone (events around each
    launch on the same stream)."""
    import numpy as np
    import torch

    import gated_delta_rule_kaczmarz_gb300 as kla
    from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS

    wl = WORKLOADS["layer_prefill"]
    inp = wl.make()
    g = {n: (x.to(dev) if isinstance(x, torch.Tensor) else x) for n, x in inp.items()}
    rng = np.random.default_rng(11)
    do = torch.from_numpy(rng.standard_normal((wl.B, wl.T, wl.H, wl.d)).astype(np.float32)).to(
        dev, torch.bfloat16)
    dST = torch.from_numpy((0.1 * rng.standard_normal((wl.B, wl.H, wl.d, wl.d))).astype(
        np.float32)).to(dev)
    ws = torch.empty(kla.kla_chunk_bwd_workspace_size(wl.B, wl.T, wl.H, wl.d), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        kla.kla_chunk_bwd(g["q"], g["k"], g["v"], g["alpha"], g["eta"], wl.eps, g["S0"], do, dST,
                          workspace=ws, stream=stream)

    for _ in range(2):
        call()
    torch.cuda.synchronize()
    n0 = kla.kla_launch_count()
    ms = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    launches = (kla.kla_launch_count() - n0) // reps
    th = wl.B * wl.T * wl.H
    # algorithmic bytes: q, k, v, d_o read and dq, dk, dv written (bf16), alpha,
    # eta read and dalpha, deta written (fp32); S0, dS_T read and dS0 written
    nbytes = th * (7 * wl.d * 2 + 4 * 4) + wl.B * wl.H * 3 * wl.d * wl.d * 4
    return dict(wl=wl, ms=sum(ms) / len(ms), bytes=nbytes, launches=launches)


def ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pk, pk_src = peaks()

    pre = time_prefill(args, world, dev)
    wl = pre["wl"]
    t_total_s = sum(pre["times"]) / 1e3
    t_total_s = max_over_ranks(t_total_s, world)
    tokens_per_step = wl.B * wl.T
    value = world * tokens_per_step * args.steps / t_total_s
    e2e_s = max_over_ranks(sum(pre["e2e_times"]) / 1e3, world)
    e2e_value = world * tokens_per_step * args.steps / e2e_s

    # roofline of the prefill call (algorithmic bytes per launch / event time)
    th = wl.B * wl.T * wl.H
    alg_bytes = th * BYTES_PER_TOKEN_HEAD + wl.B * wl.H * 2 * wl.d * wl.d * 4
    avg_s = t_total_s / args.steps
    achieved = alg_bytes / avg_s / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": TRAFFIC_PREFILL,
            "kernel": "fused_kernel (the whole prefill call)", "peak_source": pk_src,
            "algorithmic_bytes_per_launch": alg_bytes}

    dec = time_decode(args, dev, reps=args.decode_reps)
    dec_achieved = dec["bytes_per_launch"] / dec["avg_launch_s"] / 1e9
    decode = {"value": dec["steps_per_s"], "unit": "steps/s",
              "config": {"workload": "decode_b256", "B": dec["wl"].B, "H": dec["wl"].H,
                         "dk": dec["wl"].d, "dv": dec["wl"].d, "steps": dec["wl"].steps},
              "roofline": {"bound": "hbm", "achieved": dec_achieved, "peak": pk["hbm_gbs"],
                           "unit": "GB/s", "frac": dec_achieved / pk["hbm_gbs"],
                           "traffic": TRAFFIC_DECODE, "kernel": "decode_kernel",
                           "algorithmic_bytes_per_launch": dec["bytes_per_launch"]}}

    cq = time_ccq(args, dev, reps=5)
    cq_gbs = cq["bytes"] / (cq["query_ms"] / 1e3) / 1e9
    ccq = {"workload": "layer_prefill with the CCQ read (lambda ~ sigmoid(N(0,1)))",
           "query_us": cq["query_ms"] * 1e3, "layer_us": cq["layer_ms"] * 1e3,
           "layer_value": wl.B * wl.T / (cq["layer_ms"] / 1e3), "unit": "tokens/s",
           "roofline": {"bound": "hbm", "achieved": cq_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": cq_gbs / pk["hbm_gbs"], "traffic": TRAFFIC_CCQ,
                        "kernel": "fused_kernel (CCQ mode) + ccq_finish_kernel",
                        "algorithmic_bytes_per_call": cq["bytes"]}}

    bw = time_bwd(args, dev, reps=5)
    bw_gbs = bw["bytes"] / (bw["ms"] / 1e3) / 1e9
    backward = {"workload": "layer_prefill backward (d_o ~ N(0,1), dS_T ~ N(0,0.01))",
                "us": bw["ms"] * 1e3, "value": wl.B * wl.T / (bw["ms"] / 1e3), "unit": "tokens/s",
                "launches": bw["launches"],
                "roofline": {"bound": "hbm", "achieved": bw_gbs, "peak": pk["hbm_gbs"],
                             "unit": "GB/s", "frac": bw_gbs / pk["hbm_gbs"], "traffic": None,
                             "kernel": "intra_kernel + state_kernel (recording the states) + "
                                       "bwd_dstate_tc_kernel + bwd_grads_kernel",
                             "algorithmic_bytes_per_call": bw["bytes"]}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        secs, work = oracle_sample(pre["inp_cpu"], wl.B * wl.H, wl.T, cores)
        cpu = {"value": (work / wl.H) / secs, "unit": "tokens/s", "cores": min(cores, wl.B * wl.H),
               "kind": "oracle",
               "sample": f"the whole layer workload ({wl.B * wl.H} (b,h) units x {wl.T} tokens), "
                         "fp64 sequential recurrence, one thread per unit"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "layer_prefill", "B": wl.B, "T": wl.T, "H": wl.H, "dk": wl.d,
                   "dv": wl.d, "chunk": wl.chunk, "global_batch": world * wl.B,
                   "seq_len": wl.T, "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (256 MiB write)"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": pre["h2d"],
                "d2h_bytes_per_step": pre["d2h"]},
        "gpu_launches": pre["launches"],
        "clocks": pre["clocks"],
        "decode": decode,
        "ccq": ccq,
        "backward": backward,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-reps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        return reference_arm(args)
    return ours(args)


if __name__ == "__main__":
    sys.exit(main())
