"""Torch-facing helpers around the C ABI.

They allocate outputs, metadata and workspace with torch (device memory only)
and call ``pa_get_metadata`` / ``pa_decode`` / ``pa_prefill``.  All arithmetic
runs in the library's CUDA kernels.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import binding as B


def num_sms(device=None) -> int:
    return torch.cuda.get_device_properties(device or torch.cuda.current_device()).multi_processor_count


def as_bf16(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def as_f16(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 fp16 bit patterns -> torch.float16 tensor on `device`."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.float16)


def as_16(bits: np.ndarray, device, dtype: str) -> torch.Tensor:
    return as_f16(bits, device) if dtype == "f16" else as_bf16(bits, device)


def as_e4m3(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits)).to(device).view(torch.float8_e4m3fn)


@dataclass
class DecodePlan:
    shapes: B.pa_decode_shapes
    plan: B.pa_decode_plan
    meta: np.ndarray            # host copy
    meta_dev: torch.Tensor      # int32 device copy
    workspace: torch.Tensor     # uint8, zero-filled


def plan_decode(seq_lens_host, block_table_host, num_q_heads: int, num_kv_heads: int, head_dim: int,
                max_pages: int, num_pool_pages: int, kv_dtype: str = "bf16", forced_splits: int = 0,
                ctas_per_sm: int = 0, device="cuda", sms: Optional[int] = None) -> DecodePlan:
    seq_lens_host = np.asarray(seq_lens_host, dtype=np.int32)
    sh = B.pa_decode_shapes(batch=len(seq_lens_host), num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                            head_dim=head_dim, page_size=64, max_pages_per_seq=max_pages,
                            num_pool_pages=num_pool_pages,
                            kv_dtype={"bf16": B.PA_KV_BF16, "e4m3": B.PA_KV_FP8_E4M3, "f16": B.PA_KV_FP16}[kv_dtype],
                            num_sms=sms if sms is not None else num_sms(device), ctas_per_sm=ctas_per_sm,
                            forced_splits=forced_splits)
    meta, plan = B.pa_get_metadata(seq_lens_host, block_table_host, sh)
    meta_dev = torch.from_numpy(meta).to(device)
    ws = torch.zeros(max(plan.workspace_bytes, B.PA_STATUS_BYTES), dtype=torch.uint8, device=device)
    return DecodePlan(sh, plan, meta, meta_dev, ws)


def decode(p: DecodePlan, q, k_pool, v_pool, block_table, seq_lens, scale: float, k_scale=None, v_scale=None,
           out=None, lse=None, stream=None):
    sh = p.shapes
    if out is None:
        odt = torch.float16 if sh.kv_dtype == B.PA_KV_FP16 else torch.bfloat16
        out = torch.empty((sh.batch, sh.num_q_heads, sh.head_dim), dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty((sh.batch, sh.num_q_heads), dtype=torch.float32, device=q.device)
    B.pa_decode(sh, p.plan, q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, p.meta_dev, scale, out,
                lse, p.workspace, stream=stream)
    return out, lse


def prefill_shapes(batch, num_q_heads, num_kv_heads, head_dim_qk, head_dim_v, rope_dim, max_seqlen_q, total_q,
                   total_k, max_pages=0, num_pool_pages=0, device="cuda", dtype: str = "bf16") -> B.pa_prefill_shapes:
    return B.pa_prefill_shapes(batch=batch, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                               head_dim_qk=head_dim_qk, head_dim_v=head_dim_v, rope_dim=rope_dim,
                               max_seqlen_q=max_seqlen_q, total_q=total_q, total_k=total_k, page_size=64,
                               max_pages_per_seq=max_pages, num_pool_pages=num_pool_pages,
                               num_sms=num_sms(device), dtype=B.PA_KV_FP16 if dtype == "f16" else B.PA_KV_BF16)


def prefill_mla_fp8(inp, device, causal: bool = True, qo_offset=None, stream=None):
    """pa_prefill_mla_fp8 on an ``MlaE4m3Inputs`` batch (host arrays copied to
    ``device``).  Returns (out bf16, lse fp32, workspace, shapes)."""
    dev = torch.device(device)
    t8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    sh = B.pa_prefill_shapes(batch=inp.batch, num_q_heads=inp.num_q_heads, num_kv_heads=inp.num_kv_heads,
                             head_dim_qk=192, head_dim_v=128, rope_dim=64, max_seqlen_q=inp.max_seqlen_q,
                             total_q=int(inp.cu_seqlens_q[-1]), total_k=int(inp.cu_seqlens_k[-1]), page_size=64,
                             max_pages_per_seq=0, num_pool_pages=0, num_sms=num_sms(dev),
                             dtype=B.PA_KV_FP8_E4M3)
    out = torch.empty((sh.total_q, sh.num_q_heads, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((sh.total_q, sh.num_q_heads), dtype=torch.float32, device=dev)
    ws = torch.zeros(B.pa_prefill_workspace_size(sh), dtype=torch.uint8, device=dev)
    qo = qo_offset if qo_offset is not None else inp.qo_offset
    B.pa_prefill_mla_fp8(sh, t8(inp.q_nope), as_bf16(inp.q_rope, dev), t8(inp.q_scale), t8(inp.k_nope),
                         t8(inp.k_scale), as_bf16(inp.v, dev), as_bf16(inp.k_rope, dev), t8(inp.cu_seqlens_q),
                         t8(inp.cu_seqlens_k), None if qo is None else t8(np.asarray(qo, np.int32)), causal,
                         inp.scale, out, lse, ws, stream=stream)
    return out, lse, ws, sh


def prefill_mla_rope_fp8(inp, device, causal: bool = True, qo_offset=None, stream=None):
    """pa_prefill_mla_rope_fp8 on an ``MlaRopeE4m3Inputs`` batch (host arrays
    copied to ``device``).  Returns (out bf16, lse fp32, workspace, shapes)."""
    dev = torch.device(device)
    t8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    sh = B.pa_prefill_shapes(batch=inp.batch, num_q_heads=inp.num_q_heads, num_kv_heads=inp.num_kv_heads,
                             head_dim_qk=192, head_dim_v=128, rope_dim=64, max_seqlen_q=inp.max_seqlen_q,
                             total_q=int(inp.cu_seqlens_q[-1]), total_k=int(inp.cu_seqlens_k[-1]), page_size=64,
                             max_pages_per_seq=0, num_pool_pages=0, num_sms=num_sms(dev), dtype=B.PA_KV_BF16)
    out = torch.empty((sh.total_q, sh.num_q_heads, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((sh.total_q, sh.num_q_heads), dtype=torch.float32, device=dev)
    ws = torch.zeros(B.pa_prefill_mla_rope_fp8_workspace_size(sh), dtype=torch.uint8, device=dev)
    qo = qo_offset if qo_offset is not None else inp.qo_offset
    B.pa_prefill_mla_rope_fp8(sh, as_bf16(inp.q, dev), as_bf16(inp.k_nope, dev), as_bf16(inp.v, dev),
                              t8(inp.k_rope), t8(inp.k_rope_scales), t8(inp.cu_seqlens_q), t8(inp.cu_seqlens_k),
                              None if qo is None else t8(np.asarray(qo, np.int32)), causal, inp.scale, out, lse, ws,
                              stream=stream)
    return out, lse, ws, sh


def prefill(sh: B.pa_prefill_shapes, q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool = True,
            block_table=None, k_rope=None, qo_offset=None, out=None, lse=None, workspace=None, stream=None):
    dev = q.device
    if out is None:
        odt = torch.float16 if sh.dtype == B.PA_KV_FP16 else torch.bfloat16
        out = torch.empty((sh.total_q, sh.num_q_heads, sh.head_dim_v), dtype=odt, device=dev)
    if lse is None:
        lse = torch.empty((sh.total_q, sh.num_q_heads), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.zeros(B.pa_prefill_workspace_size(sh), dtype=torch.uint8, device=dev)
    B.pa_prefill(sh, q, k, v, k_rope, cu_seqlens_q, cu_seqlens_k, block_table, qo_offset, causal, scale, out, lse,
                 workspace, stream=stream)
    return out, lse, workspace
