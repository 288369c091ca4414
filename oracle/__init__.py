"""CPU oracle for attention forward over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package.  The product library never
loads it and has no CPU fallback: it shares no code with the CUDA path.

* ``decode`` / ``prefill``: fp64 attention computed directly from the
  definition in ``oracle.c`` (two-pass softmax, every element decoded exactly).
* ``scheduler``: a separate plain restatement of the split-KV scheduling rule.
* ``prefill_mla_e4m3``: the MLA prefill with per-head e4m3 q/k parts and scales.
* ``append_kv``: new tokens written into copies of the pools.
* ``bf16_to_f64`` / ``f16_to_f64`` / ``e4m3_to_f64`` / ``e4m3_from_f32``: the
  oracle's own element decoders and encoder.

Inputs are the raw bit-pattern arrays produced by the seeded generator
(``uint16`` for bf16, ``uint8`` for e4m3); outputs are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np

from . import scheduler  # noqa: F401
from .build import build as _build, LIB as _LIB

_lib = None


def _load():
    global _lib
    if _lib is None:
        _build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_decode.argtypes = [i32, i32, i32, i32, i32, i64, i32, P, P, P, P, P, P, P,
                                      dbl, P, P]
        lib.oracle_decode.restype = i32
        lib.oracle_prefill.argtypes = [i32, i32, i32, i32, i32, i32, i32, i64, P, P, P, P, P, P,
                                       P, P, i32, dbl, P, i64, P, P, i32]
        lib.oracle_prefill.restype = i32
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = dbl
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = dbl
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_double.restype = dbl
        lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.oracle_append_kv.argtypes = [i32, i32, i32, i32, i64, i32, P, P, P, P, P, P, P, P, P]
        lib.oracle_append_kv.restype = i32
        lib.oracle_prefill_mla_e4m3.argtypes = [i32, i32, i32, P, P, P, P, P, P, P, P, P, P, i32, dbl, P, i64,
                                                P, P]
        lib.oracle_prefill_mla_e4m3.restype = i32
        lib.oracle_prefill_mla_rope_e4m3.argtypes = [i32, i32, i32, P, P, P, P, P, P, P, P, i32, dbl, P, i64, P, P]
        lib.oracle_prefill_mla_rope_e4m3.restype = i32
        lib.oracle_num_threads.restype = i32
        lib.oracle_set_num_threads.argtypes = [i32]
        _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_bf16_to_double(int(x)) for x in flat]).reshape(np.shape(bits))


def f16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_f16_to_double(int(x)) for x in flat]).reshape(np.shape(bits))


def e4m3_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3_to_double(int(x)) for x in flat]).reshape(np.shape(bits))


def decode(q, k_pool, v_pool, block_table, seq_lens, scale: float, kv_dtype: str = "bf16",
           k_scale=None, v_scale=None):
    """Single-token decode.  q uint16 [B,Hq,D] (bf16, or fp16 with kv_dtype "f16");
    pools [P,Hk,64,D] (uint16 bf16/fp16 or uint8 e4m3); block_table int32
    [B,max_pages]; seq_lens int32 [B].
    Returns (out float64 [B,Hq,D], lse float64 [B,Hq])."""
    lib = _load()
    q = _c(q, np.uint16)
    kind = {"bf16": 0, "e4m3": 1, "f16": 2}[kv_dtype]
    pdt = np.uint8 if kind == 1 else np.uint16
    k_pool, v_pool = _c(k_pool, pdt), _c(v_pool, pdt)
    bt, sl = _c(block_table, np.int32), _c(seq_lens, np.int32)
    ks, vs = _c(k_scale, np.float64), _c(v_scale, np.float64)
    B, Hq, D = q.shape
    P, Hk = k_pool.shape[0], k_pool.shape[1]
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    rc = lib.oracle_decode(B, Hq, Hk, D, bt.shape[1], P, kind, _p(q), _p(k_pool), _p(v_pool),
                           _p(ks), _p(vs), _p(bt), _p(sl), float(scale), _p(out), _p(lse))
    if rc != 0:
        raise ValueError("oracle_decode: a referenced page id is out of range or "
                         "seq_len exceeds the block table")
    return out, lse


def prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool = True,
            block_table=None, k_rope=None, qo_offset=None, rows=None, dtype: str = "bf16"):
    """Chunked / ragged (optionally MLA) prefill.  See ``oracle_prefill`` in oracle.c.
    rows: optional int64 array of (token * Hq + h) to evaluate.
    Returns (out float64 [rows, Dv] or [total_q, Hq, Dv], lse)."""
    lib = _load()
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    cq, ck = _c(cu_seqlens_q, np.int32), _c(cu_seqlens_k, np.int32)
    bt = _c(block_table, np.int32)
    kr = _c(k_rope, np.uint16)
    qo = _c(qo_offset, np.int32)
    if kr is not None and bt is not None:
        raise ValueError("a shared rope key is defined for ragged keys only")
    B = len(cq) - 1
    total_q, Hq, Dqk = q.shape
    rope = 0 if kr is None else kr.shape[-1]
    Hk = k.shape[1]
    Dv = v.shape[-1]
    num_pages = k.shape[0] if bt is not None else 0
    max_pages = bt.shape[1] if bt is not None else 0
    rr = _c(rows, np.int64)
    nrows = total_q * Hq if rr is None else len(rr)
    out = np.zeros((nrows, Dv), dtype=np.float64)
    lse = np.zeros(nrows, dtype=np.float64)
    rc = lib.oracle_prefill(B, Hq, Hk, Dqk, Dv, rope, max_pages, num_pages, _p(q), _p(k), _p(v),
                            _p(kr), _p(cq), _p(ck), _p(bt), _p(qo), int(bool(causal)),
                            float(scale), _p(rr), nrows if rr is not None else 0,
                            _p(out), _p(lse), {"bf16": 0, "f16": 2}[dtype])
    if rc != 0:
        raise ValueError("oracle_prefill: a referenced page id is out of range, or a paged segment's kv_len "
                         "exceeds max_pages * 64")
    if rr is None:
        return out.reshape(total_q, Hq, Dv), lse.reshape(total_q, Hq)
    return out, lse


def e4m3_from_f32(x) -> np.ndarray:
    """The oracle's own float -> e4m3 encoder (nearest-even, saturating)."""
    lib = _load()
    flat = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.oracle_e4m3_from_float(float(v)) for v in flat], dtype=np.uint8).reshape(np.shape(x))


def append_kv(k_new, v_new, cu_new, start_pos, block_table, k_pool, v_pool, k_scale=None, v_scale=None):
    """Write new tokens into copies of the pools; returns (k_pool', v_pool').
    k_new/v_new uint16 bf16 [total_new, Hk, D]; pools [P, Hk, 64, D] uint16
    (bf16) or uint8 (e4m3, needs k_scale / v_scale float32 [Hk])."""
    lib = _load()
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)
    kind = 0 if np.asarray(k_pool).dtype == np.uint16 else 1
    kp = np.array(k_pool, copy=True, order="C")
    vp = np.array(v_pool, copy=True, order="C")
    cu, sp, bt = _c(cu_new, np.int32), _c(start_pos, np.int32), _c(block_table, np.int32)
    ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
    B = len(cu) - 1
    rc = lib.oracle_append_kv(B, kp.shape[1], kp.shape[3], bt.shape[1], kp.shape[0], kind, _p(kn), _p(vn),
                              _p(cu), _p(sp), _p(bt), _p(kp), _p(vp), _p(ks), _p(vs))
    if rc != 0:
        raise ValueError("oracle_append_kv: a position falls outside the block table or the pool")
    return kp, vp


def prefill_mla_e4m3(q_nope, q_rope, q_scale, k_nope, k_scale, v, k_rope, cu_seqlens_q, cu_seqlens_k,
                     scale: float, causal: bool = True, qo_offset=None, rows=None):
    """fp8 MLA prefill (see ``oracle_prefill_mla_e4m3`` in oracle.c).
    q_nope / k_nope uint8 e4m3 [T, H, 128]; q_rope uint16 bf16 [Tq, Hq, 64];
    k_rope uint16 bf16 [Tk, 1, 64]; v uint16 bf16 [Tk, Hk, 128]; scales float32.
    Returns (out float64 [rows, 128] or [Tq, Hq, 128], lse)."""
    lib = _load()
    qn, kn = _c(q_nope, np.uint8), _c(k_nope, np.uint8)
    qr, kr, vv = _c(q_rope, np.uint16), _c(k_rope, np.uint16), _c(v, np.uint16)
    qs, ks = _c(q_scale, np.float32), _c(k_scale, np.float32)
    cq, ck = _c(cu_seqlens_q, np.int32), _c(cu_seqlens_k, np.int32)
    qo = _c(qo_offset, np.int32)
    rr = _c(rows, np.int64)
    B = len(cq) - 1
    total_q, Hq = qn.shape[0], qn.shape[1]
    Hk = kn.shape[1]
    nrows = total_q * Hq if rr is None else len(rr)
    out = np.zeros((nrows, 128), dtype=np.float64)
    lse = np.zeros(nrows, dtype=np.float64)
    lib.oracle_prefill_mla_e4m3(B, Hq, Hk, _p(qn), _p(qr), _p(qs), _p(kn), _p(ks), _p(vv), _p(kr), _p(cq), _p(ck),
                                _p(qo), int(bool(causal)), float(scale), _p(rr), nrows if rr is not None else 0,
                                _p(out), _p(lse))
    if rr is None:
        return out.reshape(total_q, Hq, 128), lse.reshape(total_q, Hq)
    return out, lse


def prefill_mla_rope_e4m3(q, k_nope, v, k_rope, k_rope_scales, cu_seqlens_q, cu_seqlens_k, scale: float,
                          causal: bool = True, qo_offset=None, rows=None):
    """MLA prefill with an e4m3 rope key (see ``oracle_prefill_mla_rope_e4m3`` in
    oracle.c).  q uint16 bf16 [Tq, Hq, 192]; k_nope, v uint16 bf16 [Tk, Hk, 128];
    k_rope uint8 e4m3 [Tk, 1, 64] or [Tk, 64]; k_rope_scales float32 [Tk].
    Returns (out float64 [rows, 128] or [Tq, Hq, 128], lse)."""
    lib = _load()
    qq, kn, vv = _c(q, np.uint16), _c(k_nope, np.uint16), _c(v, np.uint16)
    kr, rs = _c(k_rope, np.uint8), _c(k_rope_scales, np.float32)
    cq, ck = _c(cu_seqlens_q, np.int32), _c(cu_seqlens_k, np.int32)
    qo = _c(qo_offset, np.int32)
    rr = _c(rows, np.int64)
    B = len(cq) - 1
    total_q, Hq = qq.shape[0], qq.shape[1]
    Hk = kn.shape[1]
    if kr.size != kn.shape[0] * 64 or rs.size != kn.shape[0]:
        raise ValueError("k_rope must hold 64 codes and k_rope_scales one scale per key token")
    nrows = total_q * Hq if rr is None else len(rr)
    out = np.zeros((nrows, 128), dtype=np.float64)
    lse = np.zeros(nrows, dtype=np.float64)
    lib.oracle_prefill_mla_rope_e4m3(B, Hq, Hk, _p(qq), _p(kn), _p(vv), _p(kr), _p(rs), _p(cq), _p(ck), _p(qo),
                                     int(bool(causal)), float(scale), _p(rr), nrows if rr is not None else 0,
                                     _p(out), _p(lse))
    if rr is None:
        return out.reshape(total_q, Hq, 128), lse.reshape(total_q, Hq)
    return out, lse
