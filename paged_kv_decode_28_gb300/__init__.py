"""Batched paged-KV decode attention for NVIDIA GB300 (sm_103a).

The compute path is ``libpkd.so`` (hand-written sm_103a CUDA kernels behind the
C ABI in ``include/pkd.h``); ``api`` is its Python binding.  ``workloads``
builds seeded synthetic inputs.
"""
from .api import (  # noqa: F401
    BF16, E4M3, F16, F32, Plan, PkdError, append_kv, decode_noalloc, lib, mla_decode, merge_state, merge_states, num_ctas,
    noalloc_device_errors,
    mla_units, plan_host, prefill_units, tree_units,
    single_decode, version, workspace_bytes,
)
