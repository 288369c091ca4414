"""Python binding of libpa: the C-ABI calls under the same names.

Argument marshalling only -- every step of the computation runs in the CUDA
kernels behind ``libpa.so``.  Device buffers are torch tensors (used for their
memory and stream, nothing else); host buffers are numpy arrays.  A missing
library is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pa.h")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA, PA_ERR_TIMEOUT, \
    PA_ERR_DEVICE_BOUNDS = range(7)
PA_KV_BF16, PA_KV_FP8_E4M3, PA_KV_FP16 = 0, 1, 2
PA_STATUS_BYTES = 256
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_WORKSPACE",
                4: "PA_ERR_CUDA", 5: "PA_ERR_TIMEOUT", 6: "PA_ERR_DEVICE_BOUNDS"}


class PaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class pa_decode_shapes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "max_pages_per_seq",
        "num_pool_pages", "kv_dtype", "num_sms", "ctas_per_sm", "forced_splits")]


class pa_decode_plan(ctypes.Structure):
    _fields_ = [("total_splits", ctypes.c_int32), ("num_items", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("meta_ints", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t)]


class pa_prefill_shapes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim_qk", "head_dim_v", "rope_dim", "max_seqlen_q",
        "total_q", "total_k", "page_size", "max_pages_per_seq", "num_pool_pages", "num_sms", "dtype")]


class pa_mixed_shapes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "max_pages_per_seq", "num_pool_pages",
        "kv_dtype", "num_sms", "ctas_per_sm", "forced_splits")]


class pa_mixed_plan(ctypes.Structure):
    _fields_ = [("num_decode", ctypes.c_int32), ("total_q", ctypes.c_int32), ("max_seqlen_q", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("decode", pa_decode_plan), ("workspace_bytes", ctypes.c_size_t)]


class pa_append_shapes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_kv_heads", "head_dim", "page_size", "max_pages_per_seq", "num_pool_pages", "total_new",
        "kv_dtype")]


_lib = None
_P = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """The loaded libpa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpa.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                               "or python -m paged_kv_attention_fwd_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        i32, u64, sz, f32 = ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t, ctypes.c_float
        L.pa_get_metadata.argtypes = [_P, _P, ctypes.POINTER(pa_decode_shapes), _P, sz,
                                      ctypes.POINTER(pa_decode_plan)]
        L.pa_decode.argtypes = [ctypes.POINTER(pa_decode_shapes), ctypes.POINTER(pa_decode_plan), _P, _P, _P, _P,
                                _P, _P, _P, _P, f32, _P, _P, _P, sz, _P]
        L.pa_decode_attend.argtypes = L.pa_decode.argtypes
        L.pa_decode_combine.argtypes = [ctypes.POINTER(pa_decode_shapes), ctypes.POINTER(pa_decode_plan), _P, _P,
                                        _P, _P, sz, _P]
        L.pa_decode_noalloc.argtypes = [ctypes.POINTER(pa_decode_shapes), ctypes.POINTER(pa_decode_plan), _P, _P,
                                        _P, _P, _P, _P, _P, _P, f32, _P, _P, _P, _P]
        L.pa_decode_noalloc.restype = ctypes.c_int
        L.pa_prefill.argtypes = [ctypes.POINTER(pa_prefill_shapes), _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int,
                                 f32, _P, _P, _P, sz, _P]
        L.pa_prefill_mla_fp8.argtypes = [ctypes.POINTER(pa_prefill_shapes), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                         ctypes.c_int, f32, _P, _P, _P, sz, _P]
        L.pa_prefill_mla_fp8.restype = ctypes.c_int
        L.pa_prefill_mla_rope_fp8.argtypes = [ctypes.POINTER(pa_prefill_shapes), _P, _P, _P, _P, _P, _P, _P, _P,
                                              ctypes.c_int, f32, _P, _P, _P, sz, _P]
        L.pa_prefill_mla_rope_fp8.restype = ctypes.c_int
        L.pa_prefill_mla_rope_fp8_workspace_size.argtypes = [ctypes.POINTER(pa_prefill_shapes)]
        L.pa_prefill_mla_rope_fp8_workspace_size.restype = ctypes.c_size_t
        L.pa_page_table_from_flat.argtypes = [_P, ctypes.c_int64, _P, ctypes.c_int32, ctypes.c_int32, _P, _P, sz, _P]
        L.pa_page_table_from_flat.restype = ctypes.c_int
        L.pa_get_static_plan.argtypes = [ctypes.POINTER(pa_decode_shapes), ctypes.POINTER(pa_decode_plan)]
        L.pa_get_static_plan.restype = ctypes.c_int
        L.pa_get_metadata_device.argtypes = [ctypes.POINTER(pa_decode_shapes), ctypes.POINTER(pa_decode_plan), _P, _P,
                                             _P]
        L.pa_get_metadata_device.restype = ctypes.c_int
        L.pa_get_mixed_plan.argtypes = [_P, _P, _P, ctypes.POINTER(pa_mixed_shapes), _P, sz,
                                         ctypes.POINTER(pa_mixed_plan)]
        L.pa_get_mixed_plan.restype = ctypes.c_int
        L.pa_mixed.argtypes = [ctypes.POINTER(pa_mixed_shapes), ctypes.POINTER(pa_mixed_plan), _P, _P, _P, _P, _P, _P,
                               _P, _P, f32, _P, _P, _P, sz, _P]
        L.pa_mixed.restype = ctypes.c_int
        L.pa_append_kv.argtypes = [ctypes.POINTER(pa_append_shapes), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, sz, _P]
        L.pa_append_kv.restype = ctypes.c_int
        L.pa_prefill_workspace_size.argtypes = [ctypes.POINTER(pa_prefill_shapes)]
        L.pa_prefill_workspace_size.restype = ctypes.c_size_t
        L.pa_check_status.argtypes = [_P, _P]
        L.pa_last_error.restype = ctypes.c_char_p
        L.pa_set_wait_limit_ns.argtypes = [u64]
        L.pa_set_prefill_cta_pairs.argtypes = [i32]
        L.pa_debug_wait_timeout.argtypes = [_P, u64, _P]
        L.pa_version.restype = i32
        for f in ("pa_get_metadata", "pa_decode", "pa_decode_attend", "pa_decode_combine", "pa_prefill", "pa_check_status", "pa_set_wait_limit_ns",
                  "pa_set_prefill_cta_pairs", "pa_debug_wait_timeout"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def declared_symbols() -> list:
    """Every function the public header declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:pa_status|const char\*|int32_t|size_t)\s+(pa_\w+)\s*\(", text, re.M)))


def _check(st: int) -> None:
    if st != PA_OK:
        raise PaError(st, lib().pa_last_error().decode())


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()  # torch tensor


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def pa_version() -> int:
    return lib().pa_version()


def pa_last_error() -> str:
    return lib().pa_last_error().decode()


def pa_get_metadata(seq_lens_host: np.ndarray, block_table_host: Optional[np.ndarray], shapes: pa_decode_shapes):
    """Returns (meta int32 numpy array, pa_decode_plan)."""
    sl = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
    bt = None if block_table_host is None else np.ascontiguousarray(block_table_host, dtype=np.int32)
    plan = pa_decode_plan()
    _check(lib().pa_get_metadata(_ptr(sl), _ptr(bt), ctypes.byref(shapes), None, 0, ctypes.byref(plan)))
    meta = np.zeros(plan.meta_ints, dtype=np.int32)
    _check(lib().pa_get_metadata(_ptr(sl), _ptr(bt), ctypes.byref(shapes), _ptr(meta), meta.size,
                                 ctypes.byref(plan)))
    return meta, plan


def pa_decode(shapes: pa_decode_shapes, plan: pa_decode_plan, q, k_pool, v_pool, k_scale, v_scale, block_table,
              seq_lens, meta_dev, scale: float, out, lse, workspace, workspace_bytes: Optional[int] = None,
              stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_decode(ctypes.byref(shapes), ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                           _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), _ptr(meta_dev),
                           float(scale), _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                           _stream(stream)))


def prepared(name: str, *args, stream=None):
    """A repeatable call of the C function `name` with its arguments
    marshalled once: tensors and arrays become their addresses now, structures
    are passed by reference, the stream is resolved now.  For loops that call
    one entry point on the same buffers every step (the buffers must stay
    allocated while the callable is in use).  The callable raises PaError on a
    non-OK status, like the wrappers above."""
    f = getattr(lib(), name)
    cargs = []
    for a in args:
        if isinstance(a, ctypes.Structure):
            cargs.append(ctypes.byref(a))
        elif a is None or isinstance(a, np.ndarray) or hasattr(a, "data_ptr"):
            cargs.append(_ptr(a))
        else:
            cargs.append(a)
    cargs.append(_stream(stream))
    cargs = tuple(cargs)

    def call() -> None:
        st = f(*cargs)
        if st != PA_OK:
            _check(st)

    return call


def pa_decode_attend(shapes: pa_decode_shapes, plan: pa_decode_plan, q, k_pool, v_pool, k_scale, v_scale,
                     block_table, seq_lens, meta_dev, scale: float, out, lse, workspace,
                     workspace_bytes: Optional[int] = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_attend(ctypes.byref(shapes), ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                  _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens),
                                  _ptr(meta_dev), float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                  int(workspace_bytes), _stream(stream)))


def pa_decode_combine(shapes: pa_decode_shapes, plan: pa_decode_plan, meta_dev, out, lse, workspace,
                      workspace_bytes: Optional[int] = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_combine(ctypes.byref(shapes), ctypes.byref(plan), _ptr(meta_dev), _ptr(out), _ptr(lse),
                                   _ptr(workspace), int(workspace_bytes), _stream(stream)))


def pa_decode_noalloc(shapes: pa_decode_shapes, plan: pa_decode_plan, q, k_pool, v_pool, k_scale, v_scale,
                      block_table, seq_lens, meta_dev, scale: float, out, lse, want_status: bool = True,
                      stream=None) -> int:
    """Decode without a caller workspace (the library's own 16 MiB scratch).
    Returns the device status word when want_status (the call then waits for
    the stream), else PA_OK without waiting."""
    status = ctypes.c_int32(-1)
    _check(lib().pa_decode_noalloc(ctypes.byref(shapes), ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                   _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens),
                                   _ptr(meta_dev), float(scale), _ptr(out), _ptr(lse),
                                   ctypes.byref(status) if want_status else None, _stream(stream)))
    return status.value if want_status else PA_OK


def pa_prefill(shapes: pa_prefill_shapes, q, k, v, k_rope, cu_seqlens_q, cu_seqlens_k, block_table, qo_offset,
               causal: bool, scale: float, out, lse, workspace, workspace_bytes: Optional[int] = None,
               stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_prefill(ctypes.byref(shapes), _ptr(q), _ptr(k), _ptr(v), _ptr(k_rope), _ptr(cu_seqlens_q),
                            _ptr(cu_seqlens_k), _ptr(block_table), _ptr(qo_offset), int(bool(causal)),
                            float(scale), _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                            _stream(stream)))


def pa_prefill_mla_fp8(shapes: pa_prefill_shapes, q_nope, q_rope, q_scale, k_nope, k_scale, v, k_rope, cu_seqlens_q,
                       cu_seqlens_k, qo_offset, causal: bool, scale: float, out, lse, workspace,
                       workspace_bytes: Optional[int] = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_prefill_mla_fp8(ctypes.byref(shapes), _ptr(q_nope), _ptr(q_rope), _ptr(q_scale), _ptr(k_nope),
                                    _ptr(k_scale), _ptr(v), _ptr(k_rope), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                    _ptr(qo_offset), int(bool(causal)), float(scale), _ptr(out), _ptr(lse),
                                    _ptr(workspace), int(workspace_bytes), _stream(stream)))


def pa_prefill_mla_rope_fp8(shapes: pa_prefill_shapes, q, k_nope, v, k_rope, k_rope_scales, cu_seqlens_q,
                            cu_seqlens_k, qo_offset, causal: bool, scale: float, out, lse, workspace,
                            workspace_bytes: Optional[int] = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_prefill_mla_rope_fp8(ctypes.byref(shapes), _ptr(q), _ptr(k_nope), _ptr(v), _ptr(k_rope),
                                         _ptr(k_rope_scales), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                         _ptr(qo_offset), int(bool(causal)), float(scale), _ptr(out), _ptr(lse),
                                         _ptr(workspace), int(workspace_bytes), _stream(stream)))


def pa_prefill_mla_rope_fp8_workspace_size(shapes: pa_prefill_shapes) -> int:
    return int(lib().pa_prefill_mla_rope_fp8_workspace_size(ctypes.byref(shapes)))


def pa_page_table_from_flat(kv_indices, num_indices: int, kv_lens, batch: int, max_pages_per_seq: int, block_table,
                            workspace, workspace_bytes: Optional[int] = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_page_table_from_flat(_ptr(kv_indices), int(num_indices), _ptr(kv_lens), int(batch),
                                         int(max_pages_per_seq), _ptr(block_table), _ptr(workspace),
                                         int(workspace_bytes), _stream(stream)))


def pa_get_static_plan(shapes: pa_decode_shapes) -> pa_decode_plan:
    plan = pa_decode_plan()
    _check(lib().pa_get_static_plan(ctypes.byref(shapes), ctypes.byref(plan)))
    return plan


def pa_get_metadata_device(shapes: pa_decode_shapes, static_plan: pa_decode_plan, seq_lens_dev, meta_dev,
                           stream=None) -> None:
    _check(lib().pa_get_metadata_device(ctypes.byref(shapes), ctypes.byref(static_plan), _ptr(seq_lens_dev),
                                        _ptr(meta_dev), _stream(stream)))


def pa_get_mixed_plan(cu_seqlens_q_host, kv_lens_host, block_table_host, shapes: pa_mixed_shapes):
    """Returns (decode-part metadata int32 numpy array, pa_mixed_plan)."""
    cq = np.ascontiguousarray(cu_seqlens_q_host, dtype=np.int32)
    kl = np.ascontiguousarray(kv_lens_host, dtype=np.int32)
    bt = None if block_table_host is None else np.ascontiguousarray(block_table_host, dtype=np.int32)
    plan = pa_mixed_plan()
    st = lib().pa_get_mixed_plan(_ptr(cq), _ptr(kl), _ptr(bt), ctypes.byref(shapes), None, 0, ctypes.byref(plan))
    if st not in (PA_OK, PA_ERR_WORKSPACE):
        _check(st)
    meta = np.zeros(max(plan.decode.meta_ints, 1), dtype=np.int32)
    _check(lib().pa_get_mixed_plan(_ptr(cq), _ptr(kl), _ptr(bt), ctypes.byref(shapes), _ptr(meta), meta.size,
                                   ctypes.byref(plan)))
    return meta, plan


def pa_mixed(shapes: pa_mixed_shapes, plan: pa_mixed_plan, q, k_pool, v_pool, block_table, cu_seqlens_q,
             cu_seqlens_k, kv_lens, meta_dev, scale: float, out, lse, workspace, workspace_bytes: Optional[int] = None,
             stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_mixed(ctypes.byref(shapes), ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                          _ptr(block_table), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(kv_lens), _ptr(meta_dev),
                          float(scale), _ptr(out), _ptr(lse), _ptr(workspace), int(workspace_bytes),
                          _stream(stream)))


def pa_append_kv(shapes: pa_append_shapes, k_new, v_new, cu_seqlens_new, start_pos, block_table, k_pool, v_pool,
                 k_scale, v_scale, workspace, workspace_bytes: Optional[int] = None, stream=None) -> None:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib().pa_append_kv(ctypes.byref(shapes), _ptr(k_new), _ptr(v_new), _ptr(cu_seqlens_new), _ptr(start_pos),
                              _ptr(block_table), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
                              _ptr(workspace), int(workspace_bytes), _stream(stream)))


def pa_prefill_workspace_size(shapes: pa_prefill_shapes) -> int:
    return int(lib().pa_prefill_workspace_size(ctypes.byref(shapes)))


def pa_check_status(workspace, stream=None) -> int:
    """Synchronise, read and clear the device status word; returns the pa_status code."""
    return lib().pa_check_status(_ptr(workspace), _stream(stream))


def pa_set_wait_limit_ns(limit_ns: int) -> None:
    _check(lib().pa_set_wait_limit_ns(int(limit_ns)))


def pa_set_prefill_cta_pairs(enable: bool) -> None:
    _check(lib().pa_set_prefill_cta_pairs(1 if enable else 0))


def pa_debug_wait_timeout(workspace, limit_ns: int, stream=None) -> None:
    _check(lib().pa_debug_wait_timeout(_ptr(workspace), int(limit_ns), _stream(stream)))
