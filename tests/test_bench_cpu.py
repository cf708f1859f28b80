"""The benchmark's own arithmetic, on the CPU: the algorithmic bytes and flops
of a prefill (the roofline's numerator), the choice of the bound, and the
fractions it reports.  Per token and head the chunkwise prefill reads q, k, v
and writes o (d values each) and reads alpha and eta (fp32); per (sequence,
head) it reads S0 (if given) and writes S_T (fp32); its dense-tile flops are
five C x C x d and three C x d x d products per chunk of C tokens."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6778.7, "bf16_tflops": 1876.1}


def test_bytes_and_flops_per_token_head():
    assert bench.bytes_per_token_head(128, 2) == 4 * 128 * 2 + 8 == 1032
    assert bench.bytes_per_token_head(64, 4) == 4 * 64 * 4 + 8
    C, d = 64, 128
    assert bench.flops_per_token_head(d, C) == (5 * C * C * d * 2 + 3 * C * d * d * 2) // C


def test_layer_prefill_roofline_is_the_hbm_term():
    # B4 H8 T2048 d128 bf16 with S0: 65,536 token-heads, 32 states read and written
    alg = 65536 * 1032 + 32 * 128 * 128 * 4 * 2
    assert alg == 71827456
    flops = 65536 * bench.flops_per_token_head(128)
    r = bench.roofline(alg, flops, 66.45e-6, PEAKS, "measured", None, "fused_kernel")
    assert r["bound"] == "hbm"
    assert r["t_hbm_us"] > r["t_tensor_us"]
    assert r["achieved"] == pytest.approx(alg / 66.45e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["hbm_gbs"])
    assert 0.15 < r["frac"] < 0.17


def test_the_bound_follows_the_slower_term():
    # a made-up call whose flops dominate: the tensor term is reported instead
    r = bench.roofline(1e6, 1e13, 1e-3, PEAKS, "measured", None, "k")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(1e13 / 1e-3 / 1e12 / PEAKS["bf16_tflops"])


@pytest.mark.parametrize("name,tokens", [("layer_prefill", 8192), ("long_context", 32768)])
def test_workload_algorithmic_bytes(name, tokens):
    from gated_delta_rule_kaczmarz_gb300.workloads import WORKLOADS
    wl = WORKLOADS[name]
    assert wl.B * wl.T == tokens
    th = tokens * wl.H
    units = wl.B * wl.H
    s0 = 0 if name == "long_context" else units * wl.d * wl.d * 4
    alg = th * bench.bytes_per_token_head(wl.d, 2) + s0 + units * wl.d * wl.d * 4
    expected = {"layer_prefill": 71827456, "long_context": 542113792}[name]
    assert alg == expected
