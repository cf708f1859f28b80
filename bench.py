#!/usr/bin/env python
"""Benchmark of the KLA hot path on one GB300 (or N independent replicas).

Step = one chunkwise prefill (kla_chunk_fwd) of the 0.4B-scale layer
workload: B=4, H=8, T=2048, dk=dv=128, chunk 64, bf16 q/k/v, fp32
alpha/eta/state, S0 ~ N(0,0.01), returning o and S_T.  The same run times the
two larger prefill workloads -- the 32K-token long context (B=1, H=16) and the
packed varlen batch (64 sequences, 128..8192 tokens, H=16) -- each with its own
roofline, end-to-end figure and CPU baseline, and the batched decode workload
(B=256, H=16, d=128, 64 in-place steps), the CCQ read and the backward pass.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --case NAME [--calls N] [--B B]

Timing: CUDA events on the launching stream around each step.  For the layer
workload L2 is flushed (256 MiB write) between timed steps, outside the
events; the long-context (542 MB) and varlen (4.5 GB) inputs are larger than
L2, as is the decode state (268 MB).  The end-to-end figure copies every
step's inputs from pinned host memory and its outputs back, pipelined over two
device buffer sets (copies in, compute and copies out of consecutive steps
overlap on three streams); it is the total time of all steps / steps.  For
N > 1 (torchrun) every rank runs its own replica; times are max-reduced over
ranks and value = total tokens / time.  The reference arm (--impl reference)
times the fp64 CPU oracle on the host.

--case runs one named workload a few times through the public API (a short,
fixed launch sequence for profilers; its printed time is not a benchmark
figure when run under a profiler): a prefill workload name, "decode" (single
steps on a [B, 16, 128, 128] state), "ccq" or "backward".
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
# DRAM bytes (read + write) per call from an ncu capture of the kernels as
# they are now, or None where the kernels changed after the last capture.
TRAFFIC = {"layer_prefill": 56.03e6 + 16.03e6, "long_context": None, "varlen_64": None,
           "tiny_fp32": None,
           "decode_b256": 2 * (135.83e6 + 74.59e6), "ccq": 33.90e6 + 0.12e6}
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
BYTES_PER_TOKEN_HEAD = 1032          # q,k,v,o bf16 (4 x 256 B) + alpha, eta fp32 (8 B)


def bytes_per_token_head(d: int, elem: int) -> int:
    """q, k, v read and o written (d elements of `elem` bytes each) plus
    alpha and eta (fp32): 1032 B for bf16 with d = 128 (and for fp32 with
    d = 64)."""
    return 4 * d * elem + 8
CHUNK = 64


def flops_per_token_head(d: int, chunk: int = CHUNK) -> int:
    """Dense-tile flops of the chunkwise algorithm per token and head: five
    C x C x d products and three C x d x d products per chunk."""
    return 10 * chunk * d + 6 * d * d


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def roofline(alg_bytes, flops, seconds, pk, pk_src, traffic, kernel):
    """Roofline of one call: the bound is the slower of the algorithmic bytes
    at the measured HBM copy bandwidth and the flops at the measured dense
    bf16 tensor throughput (burst); achieved and frac refer to that bound."""
    t_hbm = alg_bytes / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        bound, achieved, peak, unit = "hbm", alg_bytes / seconds / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        bound, achieved, peak, unit = ("tensor", flops / seconds / 1e12, pk["bf16_tflops"],
                                       "TFLOP/s")
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic, "kernel": kernel,
            "peak_source": pk_src, "algorithmic_bytes_per_launch": alg_bytes,
            "flops_per_launch": flops, "t_hbm_us": t_hbm * 1e6, "t_tensor_us": t_tc * 1e6}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""
    QUERY = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None

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
    tokens of a fixed-length workload; returns (seconds, token-heads)."""
    import numpy as np

    import oracle
    B, T, H, _ = inp["q"].shape
    units = [(u // H, u % H) for u in range(B * H)][:heads]
    sel = lambda x: x[[b for b, _ in units], :tokens, [h for _, h in units]][:, :, None]
    args = [sel(inp[n]).contiguous() for n in ("q", "k", "v", "alpha", "eta")]
    S0 = None if inp["S0"] is None else inp["S0"][[b for b, _ in units], [h for _, h in units]][:, None]
    # convert before timing (the oracle's input is fp64)
    conv = [np.ascontiguousarray(a.double().numpy()) for a in args]
    S0c = None if S0 is None else np.ascontiguousarray(S0.double().numpy())
    t0 = time.perf_counter()
    oracle.forward(*conv[:5], inp["eps"], S0c, nthreads=nthreads)
    return time.perf_counter() - t0, len(units) * min(tokens, T)


def oracle_sample_varlen(inp, n_seq, nthreads):
    """The fp64 oracle on the first `n_seq` packed sequences (all heads);
    returns (seconds, token-heads)."""
    import numpy as np

    import oracle
    cu = inp["cu_seqlens"].numpy()
    rows = int(cu[n_seq])
    sub = [np.ascontiguousarray(inp[n][:rows].double().numpy())
           for n in ("q", "k", "v", "alpha", "eta")]
    S0 = None if inp["S0"] is None else np.ascontiguousarray(inp["S0"][:n_seq].double().numpy())
    t0 = time.perf_counter()
    oracle.forward_varlen(*sub, inp["eps"], cu[:n_seq + 1].copy(), S0, nthreads=nthreads)
    return time.perf_counter() - t0, rows * inp["q"].shape[1]


def cpu_baseline(name, inp, wl):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload (a few seconds at most), in the workload's tokens/s."""
    cores = os.cpu_count() or 1
    if wl.kind == "varlen":
        n_seq = 4
        secs, work = oracle_sample_varlen(inp, n_seq, cores)
        used = min(cores, n_seq * wl.H)
        sample = (f"the first {n_seq} packed sequences, all {wl.H} heads "
                  f"({work // wl.H} tokens), one thread per (sequence, head)")
    elif name in ("layer_prefill", "tiny_fp32"):
        secs, work = oracle_sample(inp, wl.B * wl.H, wl.T, cores)
        used = min(cores, wl.B * wl.H)
        sample = (f"the whole {name} workload ({wl.B * wl.H} (b,h) units x {wl.T} tokens), "
                  "one thread per unit")
    else:
        units, tokens = wl.B * wl.H, 2048
        secs, work = oracle_sample(inp, units, tokens, cores)
        used = min(cores, units)
        sample = f"all {units} heads x the first {tokens} tokens, one thread per head"
    return {"value": (work / wl.H) / secs, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": sample + "; fp64 sequential recurrence"}


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


# ----------------------------------------------------------------- prefill legs
class Prefill:
    """One prefill workload on the device: inputs, outputs, workspace, and
    the public-API call on a given set of device buffers."""

    def __init__(self, name, dev):
        import torch

        import gated_delta_rule_kaczmarz_gb300 as kla
        from gated_delta_rule_kaczmarz_gb300 import binding
        from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS

        self.kla = kla
        self.name = name
        self.wl = wl = WORKLOADS[name]
        self.inp_cpu = wl.make()
        self.varlen = wl.kind == "varlen"
        q = self.inp_cpu["q"]
        self.H, self.d = wl.H, wl.d
        if self.varlen:
            self.total_T = q.shape[0]
            self.n_seq = wl.N
            self.tokens = self.total_T
            wsb = kla.kla_chunk_fwd_varlen_workspace_size(self.n_seq, self.total_T, wl.H, wl.d,
                                                          wl.d, CHUNK, binding.KLA_DTYPE_BF16)
            self.names = ("q", "k", "v", "alpha", "eta", "S0", "cu_seqlens")
        else:
            self.n_seq = wl.B
            self.tokens = wl.B * wl.T
            wsb = kla.kla_chunk_fwd_workspace_size(
                wl.B, wl.T, wl.H, wl.d, wl.d, CHUNK,
                binding.KLA_DTYPE_F32 if q.dtype == torch.float32 else binding.KLA_DTYPE_BF16)
            self.names = ("q", "k", "v", "alpha", "eta", "S0")
        self.names = tuple(n for n in self.names if self.inp_cpu[n] is not None)
        self.g = {n: self.inp_cpu[n].to(dev) for n in self.names}
        self.o = torch.empty(q.shape[:-1] + (wl.d,), dtype=q.dtype, device=dev)
        self.S_T = torch.empty((self.n_seq, wl.H, wl.d, wl.d), dtype=torch.float32, device=dev)
        self.ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
        th = self.tokens * wl.H
        units = self.n_seq * wl.H
        s0_bytes = 0 if self.inp_cpu["S0"] is None else units * wl.d * wl.d * 4
        self.alg_bytes = (th * bytes_per_token_head(wl.d, q.element_size()) + s0_bytes
                          + units * wl.d * wl.d * 4)
        self.flops = th * flops_per_token_head(wl.d)

    def call(self, d, o, S_T, stream):
        kla, wl = self.kla, self.wl
        if self.varlen:
            kla.kla_chunk_fwd_varlen(d["q"], d["k"], d["v"], d["alpha"], d["eta"], wl.eps,
                                     d["cu_seqlens"], d.get("S0"), o=o, S_T=S_T,
                                     workspace=self.ws, stream=stream)
        else:
            kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], wl.eps, d.get("S0"),
                              o=o, S_T=S_T, workspace=self.ws, stream=stream)

    def config(self, world):
        wl = self.wl
        c = {"workload": self.name, "H": wl.H, "dk": wl.d, "dv": wl.d, "chunk": wl.chunk,
             "parallelism": f"replicas x{world}"}
        if self.varlen:
            c.update(N=wl.N, total_T=self.total_T, len_range=[wl.len_lo, wl.len_hi],
                     global_batch=world * wl.N)
        else:
            c.update(B=wl.B, T=wl.T, global_batch=world * wl.B, seq_len=wl.T)
        return c


def time_device(pf, steps, warmup, flush, stream):
    """Device time of `steps` calls with resident inputs (CUDA events around
    each call on the launching stream); returns (per-call ms list, launches)."""
    import torch
    for _ in range(warmup):
        pf.call(pf.g, pf.o, pf.S_T, stream)
    torch.cuda.synchronize()
    n0 = pf.kla.kla_launch_count()
    evs = []
    for _ in range(steps):
        if flush is not None:
            flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pf.call(pf.g, pf.o, pf.S_T, stream)
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    launches = pf.kla.kla_launch_count() - n0
    return [a.elapsed_time(b) for a, b in evs], launches


def time_e2e(pf, steps, flush, stream, dev):
    """End to end through the public API from pinned host buffers: every step
    copies its own inputs in and its outputs (o, S_T) out, pipelined over two
    device buffer sets: step i+1's inputs and step i-1's outputs move on their
    own streams while step i computes.  Returns (ms per step, h2d, d2h bytes)."""
    import torch
    host = {n: pf.inp_cpu[n].pin_memory() for n in pf.names}
    nb = 2
    dbuf = [{n: torch.empty_like(pf.g[n]) for n in pf.names} for _ in range(nb)]
    obuf = [(torch.empty_like(pf.o), torch.empty_like(pf.S_T)) for _ in range(nb)]
    hout = [(torch.empty(pf.o.shape, dtype=pf.o.dtype).pin_memory(),
             torch.empty(pf.S_T.shape, dtype=pf.S_T.dtype).pin_memory()) for _ in range(nb)]
    h2d = sum(host[n].numel() * host[n].element_size() for n in pf.names)
    d2h = pf.o.numel() * pf.o.element_size() + pf.S_T.numel() * pf.S_T.element_size()
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
    for i in range(steps):
        bi = i % nb
        if i >= nb:
            s_in.wait_event(ev_done[bi])          # step i-2 finished reading these inputs
        with torch.cuda.stream(s_in):
            for n in pf.names:
                dbuf[bi][n].copy_(host[n], non_blocking=True)
            ev_in[bi].record(s_in)
        stream.wait_event(ev_in[bi])
        if i >= nb:
            stream.wait_event(ev_out[bi])         # step i-2's outputs have left
        if flush is not None:
            flush.zero_()
        pf.call(dbuf[bi], obuf[bi][0], obuf[bi][1], stream)
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
    return t_start.elapsed_time(t_end) / steps, h2d, d2h


KERNELS = {
    "layer_prefill": "fused_kernel (the whole prefill call is this one launch)",
    "long_context": "the whole call with the sequence split: intra_kernel + state_kernel_wide "
                    "(state and transition passes, one 128-column CTA per chain) + "
                    "split_combine_kernel + split_correct_kernel",
    "varlen_64": "the whole call: prep_kernel + intra_kernel + state_kernel_wide",
    "tiny_fp32": "chunk_simt_kernel (the fp32 CUDA-core chunk kernel: one launch of 4 CTAs, one "
                 "per head and 32-column block, each walking the 4 chunks in order; latency-bound "
                 "at 512 token-heads)",
}


def prefill_leg(name, args, world, dev, pk, pk_src, steps, flush_bytes, with_cpu):
    """One prefill workload: device-timed value, roofline, end-to-end and CPU
    baseline, as a dict (the headline line's fields for the layer workload)."""
    import torch
    pf = Prefill(name, dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device=dev) if flush_bytes else None
    times, launches = time_device(pf, steps, args.warmup, flush, stream)
    t_total_s = max_over_ranks(sum(times) / 1e3, world)
    value = world * pf.tokens * steps / t_total_s
    e2e_ms, h2d, d2h = time_e2e(pf, steps, flush, stream, dev)
    e2e_ms = max_over_ranks(e2e_ms, world)
    out = {
        "value": value, "unit": "tokens/s", "ms_per_step": 1e3 * t_total_s / steps,
        "steps": steps, "config": pf.config(world),
        "roofline": roofline(pf.alg_bytes, pf.flops, t_total_s / steps, pk, pk_src,
                             TRAFFIC.get(name), KERNELS[name]),
        "e2e": {"value": world * pf.tokens / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "l2": (f"flushed between timed steps ({flush_bytes >> 20} MiB write)" if flush_bytes
               else "inputs larger than L2 (no flush)"),
    }
    out["cpu_baseline"] = cpu_baseline(name, pf.inp_cpu, pf.wl) if with_cpu else None
    inp_cpu = pf.inp_cpu
    del pf
    torch.cuda.empty_cache()
    return out, inp_cpu


# ----------------------------------------------------------------- other legs
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


def replay_times(fn, reps, flush):
    """Device time of `fn` (library calls on the current stream) per call:
    captured once into a CUDA graph, then replayed with the L2 flushed before
    each timed replay, so that the host's submission time stays out of the
    device time of a call of a few microseconds.  Falls back to timing direct
    calls if the capture fails.  Returns (per-call ms list, "cuda graph" or
    "direct")."""
    import torch
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    graph, mode = None, "cuda graph"
    try:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
    except Exception:
        graph, mode = None, "direct"
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ms = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    return ms, mode


def time_ccq(args, dev, reps):
    """CCQ read-side contraction on the layer workload (bf16, B4 H8 T2048
    d128, lambda ~ sigmoid(N(0,1))): kla_ccq_query alone, and a whole CCQ
    layer (kla_ccq_query then kla_chunk_fwd on q_clean).  Inputs resident, L2
    flushed between timed calls, each call replayed from a CUDA graph."""
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
    o = torch.empty_like(g["v"])
    S_T = torch.empty_like(g["S0"])
    ws = torch.empty(max(1, kla.kla_ccq_query_workspace_size(wl.B, wl.T, wl.H, wl.d)),
                     dtype=torch.uint8, device=dev)
    fws = torch.empty(max(1, kla.kla_chunk_fwd_workspace_size(wl.B, wl.T, wl.H, wl.d, wl.d)),
                      dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def query():
        kla.kla_ccq_query(g["q"], g["k"], lam, q_clean=qc, return_stats=False, workspace=ws,
                          stream=torch.cuda.current_stream())

    def layer():
        query()
        kla.kla_chunk_fwd(qc, g["k"], g["v"], g["alpha"], g["eta"], wl.eps, g["S0"], o=o,
                          S_T=S_T, workspace=fws, stream=torch.cuda.current_stream())

    out, modes = {}, {}
    for name, f in (("query", query), ("layer", layer)):
        ms, modes[name] = replay_times(f, reps, flush)
        out[name] = sum(ms) / len(ms)
    th = wl.B * wl.T * wl.H
    # algorithmic bytes of the query: q and k read, q_clean written (bf16), lambda read
    nbytes = th * (3 * wl.d * 2 + 4)
    return dict(wl=wl, query_ms=out["query"], layer_ms=out["layer"], bytes=nbytes, timing=modes)


def time_bwd(args, dev, reps):
    """Backward pass (kla_chunk_bwd) on the layer workload (bf16, B4 H8 T2048
    d128): the gradients of sum <d_o, o> + <dS_T, S_T> with d_o ~ N(0,1) and
    dS_T ~ N(0, 0.01).  Inputs and workspace resident, L2 flushed between
    timed calls."""
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
    with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        pass
    barrier(world)
    sampler = ClockSampler(bus).start()
    time.sleep(0.3)
    # headline: the layer workload (the configuration the metric's first
    # clause is quoted on: one 0.4B-scale layer); then the two larger ones
    head, cpu_inputs = prefill_leg("layer_prefill", args, world, dev, pk, pk_src, args.steps,
                                   256 << 20, False)
    cpu_inputs = {"layer_prefill": cpu_inputs}
    legs = {}
    for name in ("long_context", "varlen_64"):
        legs[name], cpu_inputs[name] = prefill_leg(name, args, world, dev, pk, pk_src,
                                                   args.big_steps, 0, False)
    # the small fp32 correctness workload (inputs far below L2: flushed)
    legs["tiny_fp32"], cpu_inputs["tiny_fp32"] = prefill_leg(
        "tiny_fp32", args, world, dev, pk, pk_src, args.steps, 256 << 20, False)

    dec = time_decode(args, dev, reps=args.decode_reps)
    cq = time_ccq(args, dev, reps=5)
    bw = time_bwd(args, dev, reps=5)
    clocks = sampler.stop()
    barrier(world)

    # CPU baselines after every GPU measurement (the oracle is never timed
    # inside a GPU region)
    if with_cpu:
        from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS
        head["cpu_baseline"] = cpu_baseline("layer_prefill", cpu_inputs["layer_prefill"],
                                            WORKLOADS["layer_prefill"])
        for name in legs:
            legs[name]["cpu_baseline"] = cpu_baseline(name, cpu_inputs[name], WORKLOADS[name])
    del cpu_inputs

    dec_achieved = dec["bytes_per_launch"] / dec["avg_launch_s"] / 1e9
    decode = {"value": dec["steps_per_s"], "unit": "steps/s",
              "config": {"workload": "decode_b256", "B": dec["wl"].B, "H": dec["wl"].H,
                         "dk": dec["wl"].d, "dv": dec["wl"].d, "steps": dec["wl"].steps},
              "roofline": {"bound": "hbm", "achieved": dec_achieved, "peak": pk["hbm_gbs"],
                           "unit": "GB/s", "frac": dec_achieved / pk["hbm_gbs"],
                           "traffic": TRAFFIC["decode_b256"], "kernel": "decode_kernel",
                           "algorithmic_bytes_per_launch": dec["bytes_per_launch"]}}
    wl = dec["wl"]
    cq_gbs = cq["bytes"] / (cq["query_ms"] / 1e3) / 1e9
    lw = cq["wl"]
    ccq = {"workload": "layer_prefill with the CCQ read (lambda ~ sigmoid(N(0,1)))",
           "query_us": cq["query_ms"] * 1e3, "layer_us": cq["layer_ms"] * 1e3,
           "timing": cq["timing"],
           "layer_value": lw.B * lw.T / (cq["layer_ms"] / 1e3), "unit": "tokens/s",
           "roofline": {"bound": "hbm", "achieved": cq_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": cq_gbs / pk["hbm_gbs"], "traffic": TRAFFIC["ccq"],
                        "kernel": "ccq_query_tc_kernel",
                        "algorithmic_bytes_per_call": cq["bytes"]}}
    bw_gbs = bw["bytes"] / (bw["ms"] / 1e3) / 1e9
    backward = {"workload": "layer_prefill backward (d_o ~ N(0,1), dS_T ~ N(0,0.01))",
                "us": bw["ms"] * 1e3, "value": lw.B * lw.T / (bw["ms"] / 1e3), "unit": "tokens/s",
                "launches": bw["launches"],
                "roofline": {"bound": "hbm", "achieved": bw_gbs, "peak": pk["hbm_gbs"],
                             "unit": "GB/s", "frac": bw_gbs / pk["hbm_gbs"], "traffic": None,
                             "kernel": "intra_kernel + state_kernel (recording the states) + "
                                       "bwd_dstate_tc_kernel + bwd_grads_tc_kernel",
                             "algorithmic_bytes_per_call": bw["bytes"]}}

    cfg = head["config"]
    cfg["l2"] = head["l2"]
    cfg["why_this_workload"] = ("the metric quotes prefill on one 0.4B-scale layer (B4 H8 "
                                "T2048); the 32K-token long context and the 300K-token varlen "
                                "batch are reported under long_context and varlen_64")
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": cfg,
        "roofline": head["roofline"],
        "cpu_baseline": head["cpu_baseline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": clocks,
        "long_context": legs["long_context"],
        "varlen_64": legs["varlen_64"],
        "tiny_fp32": legs["tiny_fp32"],
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


# ----------------------------------------------------------------- --case
def run_case(args) -> int:
    """A few calls of one named workload through the public API on cuda:0
    (inputs uploaded first); prints the mean time per call."""
    import torch

    import gated_delta_rule_kaczmarz_gb300 as kla
    from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS, decode_inputs

    def dev(inp):
        return {n: (x.cuda() if isinstance(x, torch.Tensor) else x) for n, x in inp.items()}

    calls = []
    if args.case == "backward":
        wl = WORKLOADS["layer_prefill"]
        inp = dev(wl.make())
        gen = torch.Generator(device="cuda").manual_seed(11)
        do = torch.randn((wl.B, wl.T, wl.H, wl.d), device="cuda", generator=gen).to(torch.bfloat16)
        dST = 0.1 * torch.randn((wl.B, wl.H, wl.d, wl.d), device="cuda", generator=gen)
        ws = torch.empty(kla.kla_chunk_bwd_workspace_size(wl.B, wl.T, wl.H, wl.d),
                         dtype=torch.uint8, device="cuda")
        calls = [lambda: kla.kla_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["eta"],
                                           wl.eps, inp["S0"], do, dST, workspace=ws)] * args.calls
    elif args.case == "ccq":
        inp = dev(WORKLOADS["layer_prefill"].make())
        lam = torch.full(inp["eta"].shape, 0.5, dtype=torch.float32, device="cuda")
        calls = [lambda: kla.kla_ccq_query(inp["q"], inp["k"], lam)] * args.calls
    elif args.case == "decode":
        inp = dev(decode_inputs(args.B, 16, 128, 128, steps=args.calls, dtype="bf16", seed=3))
        S = inp["S"]
        o = torch.empty_like(inp["v"][0])
        for t in range(args.calls):
            calls.append(lambda t=t: kla.kla_decode_step(
                inp["q"][t], inp["k"][t], inp["v"][t], inp["alpha"][t], inp["eta"][t],
                inp["eps"], S, o=o))
    elif args.case in WORKLOADS:
        pf = Prefill(args.case, torch.device("cuda", 0))
        stream = torch.cuda.current_stream()
        calls = [lambda: pf.call(pf.g, pf.o, pf.S_T, stream)] * args.calls
    else:
        raise SystemExit(f"unknown case {args.case}")
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for c in calls:
        c()
    e1.record()
    torch.cuda.synchronize()
    print(f"{args.case}: {len(calls)} calls, "
          f"{e0.elapsed_time(e1) * 1e3 / max(1, len(calls)):.1f} us/call")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--big-steps", type=int, default=10,
                    help="timed calls of the long-context and varlen workloads")
    ap.add_argument("--decode-reps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", help="run one named workload a few times (for profilers)")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--B", type=int, default=128, help="batch of the decode case")
    args = ap.parse_args()
    if args.case:
        return run_case(args)
    if args.impl == "reference":
        return reference_arm(args)
    return ours(args)


if __name__ == "__main__":
    sys.exit(main())
