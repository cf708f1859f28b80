"""CPU-only checks of the C ABI: the library builds and loads, exports every
symbol include/kla.h declares, and rejects bad requests on the host before
any device work.  No compute call is made (there is no GPU here)."""
import ctypes
import os
import re

import pytest
import torch

import gated_delta_rule_kaczmarz_gb300 as kla
from gated_delta_rule_kaczmarz_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kla.h")

no_gpu_only = pytest.mark.skipif(torch.cuda.is_available(),
                                 reason="uses fake device pointers; host validation only")


def declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"KLA_API\s+[\w\s\*]*?\b(kla_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    syms = declared_symbols()
    for name in ("kla_chunk_fwd", "kla_chunk_fwd_varlen", "kla_decode_step",
                 "kla_status_str", "kla_workspace_status"):
        assert name in syms


def test_library_exports_every_declared_symbol():
    lib = binding.load()
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_binding_names_match_the_abi():
    for name in declared_symbols():
        if name == "kla_last_error_message":
            continue
        assert hasattr(kla, name) or hasattr(binding, name), name


def test_status_strings_and_version():
    assert kla.kla_status_str(0) == "ok"
    assert "unsupported" in kla.kla_status_str(2)
    assert kla.kla_status_str(99) == "unknown status"
    assert kla.kla_version() >= 100


def test_workspace_sizes():
    assert kla.kla_chunk_fwd_workspace_size(1, 256, 2, 96, 96, 64, binding.KLA_DTYPE_F32) == 0
    assert kla.kla_chunk_fwd_workspace_size(1, 256, 2, 64, 64, 32, binding.KLA_DTYPE_F32) == 0
    # varlen always carries a status word
    assert kla.kla_chunk_fwd_varlen_workspace_size(3, 100, 2, 64, 64, 64,
                                                   binding.KLA_DTYPE_F32) >= 256


FAKE = 0x10000  # aligned, never dereferenced: validation fails first


def _call_chunk(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, alpha=FAKE, eta=FAKE, eps=1e-6, S0=None, o=FAKE, S_T=None,
             B=1, T=64, H=1, dk=64, dv=64, chunk=64, dtype=0, ws=None, wsb=0, stream=None)
    a.update(over)
    return lib.kla_chunk_fwd(a["q"], a["k"], a["v"], a["alpha"], a["eta"], a["eps"], a["S0"],
                             a["o"], a["S_T"], a["B"], a["T"], a["H"], a["dk"], a["dv"],
                             a["chunk"], a["dtype"], a["ws"], a["wsb"], a["stream"])


@no_gpu_only
@pytest.mark.parametrize("over,status", [
    (dict(dk=96, dv=96), binding.KLA_ERR_UNSUPPORTED),
    (dict(dk=64, dv=128), binding.KLA_ERR_UNSUPPORTED),
    (dict(chunk=32), binding.KLA_ERR_UNSUPPORTED),
    (dict(B=-1), binding.KLA_ERR_INVALID_ARG),
    (dict(H=0), binding.KLA_ERR_INVALID_ARG),
    (dict(dtype=7), binding.KLA_ERR_INVALID_ARG),
    (dict(q=None), binding.KLA_ERR_INVALID_ARG),
    (dict(o=None), binding.KLA_ERR_INVALID_ARG),
    (dict(k=FAKE + 2), binding.KLA_ERR_INVALID_ARG),
    (dict(alpha=FAKE + 2), binding.KLA_ERR_INVALID_ARG),
    (dict(eps=-1.0), binding.KLA_ERR_INVALID_ARG),
])
def test_chunk_fwd_host_validation(over, status):
    lib = binding.load()
    assert _call_chunk(lib, **over) == status
    assert lib.kla_last_error_message().decode() != ""


@no_gpu_only
def test_varlen_host_validation():
    lib = binding.load()
    f = lib.kla_chunk_fwd_varlen
    # N == 0 with tokens is inconsistent
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, None, FAKE, None, FAKE, 0, 10, 1, 64, 64, 64, 0,
             None, 0, None) == binding.KLA_ERR_INVALID_ARG
    # missing cu_seqlens
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, None, FAKE, None, None, 2, 10, 1, 64, 64, 64, 0,
             None, 0, None) == binding.KLA_ERR_INVALID_ARG
    # missing workspace (varlen always needs the status word)
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, None, FAKE, None, FAKE, 2, 10, 1, 64, 64, 64, 0,
             None, 0, None) == binding.KLA_ERR_WORKSPACE
    # workspace misaligned
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, None, FAKE, None, FAKE, 2, 10, 1, 64, 64, 64, 0,
             FAKE + 16, 4096, None) == binding.KLA_ERR_INVALID_ARG


@no_gpu_only
def test_decode_host_validation():
    lib = binding.load()
    f = lib.kla_decode_step
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, FAKE, FAKE, 2, 2, 80, 80, 1, None) == \
        binding.KLA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, None, FAKE, 2, 2, 64, 64, 1, None) == \
        binding.KLA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, FAKE + 4, FAKE, 2, 2, 64, 64, 1, None) == \
        binding.KLA_ERR_INVALID_ARG
    # B == 0 is a valid no-op
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, FAKE, FAKE, 0, 2, 64, 64, 1, None) == binding.KLA_OK


@no_gpu_only
def test_injected_launch_fault_is_reported_without_device_work(monkeypatch):
    lib = binding.load()
    monkeypatch.setenv("KLA_FAULT_INJECT", "launch")
    assert lib.kla_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, FAKE, FAKE, 2, 2, 64, 64, 1,
                               None) == binding.KLA_ERR_CUDA
    assert "injected" in lib.kla_last_error_message().decode()
    assert _call_chunk(lib) == binding.KLA_ERR_CUDA
    assert "injected" in lib.kla_last_error_message().decode()


def test_workspace_status_without_workspace_is_ok():
    lib = binding.load()
    assert lib.kla_workspace_status(None, 0, None) == binding.KLA_OK


def test_binding_raises_on_cpu_tensors():
    q = torch.zeros(1, 64, 1, 64)
    with pytest.raises(ValueError):
        kla.kla_chunk_fwd(q, q, q, torch.ones(1, 64, 1), torch.ones(1, 64, 1), 1e-6)


@no_gpu_only
def test_unknown_beta_mode_is_rejected_before_device_work():
    lib = binding.load()
    assert lib.kla_chunk_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, None, FAKE, None, 1, 64, 1,
                                64, 64, 64, 0, 2, None, 0, None) == binding.KLA_ERR_INVALID_ARG
    assert lib.kla_chunk_fwd_varlen_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, None, FAKE, None, FAKE,
                                       2, 10, 1, 64, 64, 64, 0, -1, None, 0, None) == \
        binding.KLA_ERR_INVALID_ARG
    assert lib.kla_decode_step_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, FAKE, FAKE, 2, 2, 64, 64, 1,
                                  9, None) == binding.KLA_ERR_INVALID_ARG
    assert "beta_mode" in lib.kla_last_error_message().decode()


@no_gpu_only
def test_ccq_host_validation():
    lib = binding.load()
    f = lib.kla_ccq_query
    # dk 96 unsupported
    assert f(FAKE, FAKE, FAKE, None, None, None, FAKE, None, None, None, 1, 64, 1, 96, 1,
             None, 0, None) == binding.KLA_ERR_UNSUPPORTED
    # missing q
    assert f(None, FAKE, FAKE, None, None, None, FAKE, None, None, None, 1, 64, 1, 64, 1,
             None, 0, None) == binding.KLA_ERR_INVALID_ARG
    # missing workspace
    assert f(FAKE, FAKE, FAKE, None, None, None, FAKE, None, None, None, 1, 64, 1, 64, 1,
             None, 0, None) == binding.KLA_ERR_WORKSPACE
    # workspace not 256-byte aligned
    assert f(FAKE, FAKE, FAKE, None, None, None, FAKE, None, None, None, 1, 64, 1, 64, 1,
             ctypes.c_void_p(0x10010), 1 << 30, None) == binding.KLA_ERR_INVALID_ARG
    assert "aligned" in lib.kla_last_error_message().decode()
    assert lib.kla_ccq_query_workspace_size(1, 64, 1, 64, 1) > 0
    # the tensor-core path (bf16, dk 128) keeps nothing but the status word
    assert lib.kla_ccq_query_workspace_size(2, 256, 2, 128, 1) == 256
    g = lib.kla_ccq_query_step
    assert g(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 2, 2, 64, 1, None) == \
        binding.KLA_ERR_INVALID_ARG
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 2, 64, 1, None) == binding.KLA_OK


@no_gpu_only
def test_backward_host_validation():
    lib = binding.load()
    f = lib.kla_chunk_bwd
    base = [FAKE, FAKE, FAKE, FAKE, FAKE, 1e-6, None, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE,
            None, 1, 64, 1, 64, 64, 64, 1, 0]
    def call(over=None, ws=None, wsb=0):
        a = list(base)
        for i, x in (over or {}).items():
            a[i] = x
        return f(*a, ws, wsb, None)
    # missing workspace
    assert call() == binding.KLA_ERR_WORKSPACE
    # dalpha without alpha
    assert call({3: None}) == binding.KLA_ERR_INVALID_ARG
    assert "dalpha" in lib.kla_last_error_message().decode()
    # unknown beta mode, unsupported head size, missing d_o
    assert call({22: 7}) == binding.KLA_ERR_INVALID_ARG
    assert call({18: 96, 19: 96}) == binding.KLA_ERR_UNSUPPORTED
    assert call({7: None}, ctypes.c_void_p(0x100000), 1 << 40) == binding.KLA_ERR_INVALID_ARG
    # misaligned workspace
    assert call(None, ctypes.c_void_p(0x100010), 1 << 40) == binding.KLA_ERR_INVALID_ARG
    n = lib.kla_chunk_bwd_workspace_size(1, 64, 1, 64, 1)
    assert n >= 2 * 64 * 64 * 4


def test_sequence_split_workspace(monkeypatch):
    """The split's buffers (per-segment end states, transitions, the
    correction rows, the start states) enlarge the forward's workspace; a
    factor above the sequence's count of 128-token tiles is ignored."""
    lib = binding.load()
    size = lambda: lib.kla_chunk_fwd_workspace_size(1, 32768, 16, 128, 128, 64, 1)
    monkeypatch.setenv("KLA_SEQ_SPLIT", "1")
    base = size()
    monkeypatch.setenv("KLA_SEQ_SPLIT", "2")
    split2 = size()
    # correction rows alone: T * H * 128 bf16
    assert split2 - base >= 32768 * 16 * 128 * 2
    monkeypatch.setenv("KLA_SEQ_SPLIT", "3")   # segments of 86 + 85 + 85 tiles
    assert size() > base
    small = lambda: lib.kla_chunk_fwd_workspace_size(1, 256, 16, 128, 128, 64, 1)
    monkeypatch.setenv("KLA_SEQ_SPLIT", "1")
    small_base = small()
    monkeypatch.setenv("KLA_SEQ_SPLIT", "3")   # 256 tokens: two tiles
    assert small() == small_base


def test_default_split_choice(monkeypatch):
    """The default split factor, seen through the workspace size (which
    depends on it): the long-context shape (B1 H16 T32768) takes five
    segments of unequal length (16 x 9 chains fit one 128-column CTA each on
    148-152 SMs, six would not), the layer shape (B4 H8 T2048) no split."""
    lib = binding.load()
    def size(B, T, H, P=None):
        if P is None:
            monkeypatch.delenv("KLA_SEQ_SPLIT", raising=False)
        else:
            monkeypatch.setenv("KLA_SEQ_SPLIT", str(P))
        return lib.kla_chunk_fwd_workspace_size(B, T, H, 128, 128, 64, 1)
    long_default = size(1, 32768, 16)
    assert long_default == size(1, 32768, 16, 5)
    assert long_default != size(1, 32768, 16, 4)
    assert long_default != size(1, 32768, 16, 6)
    assert size(4, 2048, 8) == size(4, 2048, 8, 1)
    # two heads of 32K tokens: eight equal segments (60 chains of two CTAs)
    assert size(1, 32768, 2) == size(1, 32768, 2, 8)
    # B2 H4 T8192: five unequal segments of 13 + 13 + 13 + 13 + 12 tiles, two
    # 64-column CTAs per chain (8 x 9 chains, 144 CTAs)
    assert size(2, 8192, 4) == size(2, 8192, 4, 5)
    assert size(2, 8192, 4) != size(2, 8192, 4, 4)
