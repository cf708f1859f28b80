"""Kaczmarz Linear Attention (KLA) for NVIDIA GB300 (sm_103a).

The compute path is the CUDA library ``libkla_gb300.so`` (C ABI in
``include/kla.h``); ``binding`` is its thin ctypes binding.  ``workloads``
draws seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    KlaError,
    kla_ccq_query,
    kla_ccq_query_step,
    kla_ccq_query_workspace_size,
    kla_chunk,
    kla_chunk_bwd,
    kla_chunk_bwd_varlen,
    kla_chunk_bwd_varlen_workspace_size,
    kla_chunk_bwd_workspace_size,
    kla_chunk_fwd,
    kla_chunk_fwd_ex,
    kla_chunk_fwd_noalloc,
    kla_chunk_fwd_noalloc_status,
    kla_chunk_fwd_varlen,
    kla_chunk_fwd_varlen_ex,
    kla_chunk_fwd_varlen_workspace_size,
    kla_chunk_fwd_workspace_size,
    kla_decode_step,
    kla_decode_step_ex,
    kla_launch_count,
    kla_status_str,
    kla_version,
    kla_workspace_status,
    load,
)
