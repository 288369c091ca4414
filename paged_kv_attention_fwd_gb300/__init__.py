"""Attention forward over a paged KV cache for GB300 (sm_103a).

The computation lives in ``libpa.so`` (hand-written CUDA kernels behind a C
ABI, declared in ``include/pa.h``); ``binding`` exposes those calls to Python
under the same names, and ``ops`` wraps them for torch tensors.  ``workloads``
builds seeded synthetic inputs.  Nothing here computes attention on the CPU.
"""
from .binding import (  # noqa: F401  (the C-ABI calls, constants and structs)
    PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA, PA_ERR_TIMEOUT,
    PA_ERR_DEVICE_BOUNDS, PA_KV_BF16, PA_KV_FP8_E4M3, PA_KV_FP16, PA_STATUS_BYTES, PaError,
    pa_decode_shapes, pa_decode_plan, pa_prefill_shapes, pa_mixed_shapes, pa_mixed_plan, pa_append_shapes,
    pa_version, pa_last_error, pa_check_status, pa_set_wait_limit_ns, pa_set_prefill_cta_pairs,
    pa_debug_wait_timeout,
    pa_get_metadata, pa_get_static_plan, pa_get_metadata_device, pa_page_table_from_flat,
    pa_decode, pa_decode_attend, pa_decode_combine, pa_decode_noalloc,
    pa_prefill, pa_prefill_workspace_size, pa_prefill_mla_fp8, pa_prefill_mla_rope_fp8,
    pa_prefill_mla_rope_fp8_workspace_size, pa_get_mixed_plan, pa_mixed, pa_append_kv,
)

__version__ = "0.1.0"
