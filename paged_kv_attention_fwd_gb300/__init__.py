"""Attention forward over a paged KV cache for GB300 (sm_103a).

The computation lives in ``libpa.so`` (hand-written CUDA kernels behind a C
ABI, declared in ``include/pa.h``); ``binding`` exposes those calls to Python
under the same names, and ``ops`` wraps them for torch tensors.  ``workloads``
builds seeded synthetic inputs.  Nothing here computes attention on the CPU.
"""
from .binding import (  # noqa: F401
    PaError, pa_append_kv, pa_append_shapes, pa_check_status, pa_get_mixed_plan, pa_mixed, pa_mixed_plan,
    pa_mixed_shapes, pa_debug_wait_timeout, pa_decode, pa_decode_attend, pa_decode_combine, pa_decode_plan, pa_decode_shapes,
    pa_get_metadata, pa_get_metadata_device, pa_get_static_plan, pa_last_error, pa_prefill, pa_prefill_shapes, pa_set_wait_limit_ns, pa_version,
    PA_KV_BF16, PA_KV_FP8_E4M3, PA_STATUS_BYTES,
)

__version__ = "0.1.0"
