"""Seeded synthetic inputs for paged KV attention forward.

This module builds what a caller hands to the library -- query rows, paged K/V
pools, block tables, sequence lengths, ragged offsets -- from a seed, with the
shapes and value distributions of the workloads described on the FlashMLA
"Tensor Shapes Reference" page (section "Function Reference") and the MATE
``msa_interface`` module (``_build_page_table_from_flat_kv_indices``,
``_make_cu_seqlens``).  It holds none of the attention arithmetic: no scores,
no softmax, no gather through the block table.  Both the CUDA path and the CPU
oracle are fed from here, and neither is imported by it.

Element encodings returned here are raw bit patterns so that both consumers
decode them on their own:
  * bf16  -> numpy ``uint16`` (the upper half of an IEEE fp32 word),
  * e4m3  -> numpy ``uint8`` (OCP FP8 E4M3, "fn" variant: no infinities).

Random numbers: every tensor is drawn from its own stream
``(seed, stream_id, chunk)`` of numpy's PCG64 generator, in fixed-size chunks,
so the values do not depend on how many threads fill them.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

PAGE_SIZE = 64
_CHUNK = 1 << 22

# stream ids: one per tensor role, so adding a tensor never shifts another
_S_SEQLENS, _S_PERM, _S_Q, _S_K, _S_V, _S_KROPE, _S_PREFIX, _S_QROPE = 1, 2, 3, 4, 5, 6, 7, 8


def _rng(seed: int, stream: int, chunk: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, chunk])))


def normal_f32(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard-normal float32 values, filled chunk by chunk in threads."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def fill(c: int) -> None:
        lo = c * _CHUNK
        hi = min(n, lo + _CHUNK)
        _rng(seed, stream, c).standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    if nchunks <= 1:
        if n:
            fill(0)
    else:
        with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 4)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


E4M3_MAX = 448.0


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Encode to OCP FP8 E4M3 (bias 7, 3 mantissa bits, max 448, no inf).

    Rounds to nearest with ties to even and saturates to +-448 (finite inputs).
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # exponent of the binade, floored at the subnormal exponent -6
    _, e2 = np.frexp(a)              # a = f * 2**e2 with f in [0.5, 1)
    e = np.maximum(e2 - 1, -6)       # a in [2**e, 2**(e+1))
    quantum = np.ldexp(1.0, e - 3)   # 3 mantissa bits
    q = np.rint(a / quantum) * quantum
    q = np.minimum(q, E4M3_MAX)
    # encode q (exactly representable now)
    _, qe2 = np.frexp(q)
    qe = qe2 - 1
    normal = q >= 2.0 ** -6
    exp_field = np.where(normal, qe + 7, 0)
    mant = np.where(normal, q / np.ldexp(1.0, qe) - 1.0, q / 2.0 ** -9)
    mant = np.where(normal, mant * 8.0, mant)
    bits = (exp_field.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    bits = np.where(q == 0, 0, bits)
    bits = bits | (sign.astype(np.int64) << 7)
    return bits.astype(np.uint8)


def bf16_normal(seed: int, stream: int, shape) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    return f32_to_bf16_bits(normal_f32(seed, stream, n)).reshape(shape)


def f16_normal(seed: int, stream: int, shape) -> np.ndarray:
    """N(0,1) rounded to IEEE fp16 (nearest even); uint16 bit patterns."""
    n = int(np.prod(shape)) if len(shape) else 1
    return normal_f32(seed, stream, n).astype(np.float16).view(np.uint16).reshape(shape)


def normal_16(seed: int, stream: int, shape, dtype: str) -> np.ndarray:
    return f16_normal(seed, stream, shape) if dtype == "f16" else bf16_normal_fast(seed, stream, shape)


def cu_seqlens(lengths: np.ndarray) -> np.ndarray:
    """int32 [n+1] running offsets of ragged segments (first entry 0)."""
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return out.astype(np.int32)


def pages_for(length: int, page_size: int = PAGE_SIZE) -> int:
    return (int(length) + page_size - 1) // page_size


def assign_pages(seq_lens: np.ndarray, seed: int, extra_pages: int = 0,
                 max_pages: Optional[int] = None, page_size: int = PAGE_SIZE):
    """Shuffled physical page ids handed to each sequence in order.

    Returns (block_table int32 [B, max_pages], num_pool_pages).  The pool holds
    sum(ceil(len/64)) + extra_pages pages; physical ids are a seeded
    permutation; unused block_table entries are 0 (as the MATE page-table
    builder pads).
    """
    counts = [pages_for(s, page_size) for s in seq_lens]
    total = sum(counts)
    num_pool = total + extra_pages
    if max_pages is None:
        max_pages = max(counts) if counts else 0
    max_pages = max(max_pages, 1)
    perm = _rng(seed, _S_PERM).permutation(num_pool).astype(np.int32)
    bt = np.zeros((len(seq_lens), max_pages), dtype=np.int32)
    pos = 0
    for b, c in enumerate(counts):
        bt[b, :c] = perm[pos:pos + c]
        pos += c
    return bt, num_pool


@dataclass
class DecodeInputs:
    q: np.ndarray            # uint16 bf16 bits [B, Hq, D]
    k_pool: np.ndarray       # uint16 [P, Hk, 64, D] (bf16) or uint8 (e4m3)
    v_pool: np.ndarray
    block_table: np.ndarray  # int32 [B, max_pages]
    seq_lens: np.ndarray     # int32 [B]
    scale: float
    kv_dtype: str            # "bf16" | "e4m3" | "f16" (fp16 q and pools)
    k_scale: Optional[np.ndarray] = None   # float32 [Hk] (e4m3 only)
    v_scale: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)

    @property
    def batch(self): return self.q.shape[0]
    @property
    def num_q_heads(self): return self.q.shape[1]
    @property
    def head_dim(self): return self.q.shape[2]
    @property
    def num_kv_heads(self): return self.k_pool.shape[1]
    @property
    def num_pool_pages(self): return self.k_pool.shape[0]
    @property
    def max_pages(self): return self.block_table.shape[1]


def _to_bf16_bits_fast(x: np.ndarray) -> np.ndarray:
    """Same result as f32_to_bf16_bits (round to nearest even), via torch's
    multi-threaded CPU cast; used for the large pools."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _to_e4m3_bits_fast(x: np.ndarray) -> np.ndarray:
    """Same result as f32_to_e4m3_bits for inputs already inside [-448, 448]."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def bf16_normal_fast(seed: int, stream: int, shape) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    return _to_bf16_bits_fast(normal_f32(seed, stream, n)).reshape(shape)


def quantise_per_head(x: np.ndarray, fast: bool = True):
    """x float32 [P, Hk, 64, D] -> (e4m3 bits, float32 scale per KV head).

    scale_h = amax(|x[:, h]|) / 448 (1 for an all-zero head); the stored code is
    e4m3(clamp(float32(x / scale_h), -448, 448)), rounded to nearest even.
    """
    import torch
    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    hk = x.shape[1]
    amax = xt.abs().amax(dim=(0, 2, 3)) if x.shape[0] else torch.zeros(hk)
    scales = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    y = (xt / scales.view(1, hk, 1, 1)).clamp_(-E4M3_MAX, E4M3_MAX)
    bits = _to_e4m3_bits_fast(y.numpy()) if fast else f32_to_e4m3_bits(y.numpy())
    return bits.reshape(x.shape), scales.numpy()


def make_decode(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                seq_lens, seed: int = 0, kv_dtype: str = "bf16",
                extra_pages: int = 0, max_pages: Optional[int] = None) -> DecodeInputs:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert len(seq_lens) == batch
    bt, num_pool = assign_pages(seq_lens, seed, extra_pages, max_pages)
    pool_shape = (num_pool, num_kv_heads, PAGE_SIZE, head_dim)
    q = (f16_normal if kv_dtype == "f16" else bf16_normal)(seed, _S_Q, (batch, num_q_heads, head_dim))
    n = int(np.prod(pool_shape))
    if kv_dtype in ("bf16", "f16"):
        k = normal_16(seed, _S_K, pool_shape, kv_dtype)
        v = normal_16(seed, _S_V, pool_shape, kv_dtype)
        ks = vs = None
    elif kv_dtype == "e4m3":
        k, ks = quantise_per_head(normal_f32(seed, _S_K, n).reshape(pool_shape))
        v, vs = quantise_per_head(normal_f32(seed, _S_V, n).reshape(pool_shape))
    else:
        raise ValueError(kv_dtype)
    return DecodeInputs(q=q, k_pool=k, v_pool=v, block_table=bt, seq_lens=seq_lens,
                        scale=1.0 / math.sqrt(head_dim), kv_dtype=kv_dtype,
                        k_scale=ks, v_scale=vs)


def uniform_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] inclusive."""
    return _rng(seed, _S_SEQLENS).integers(lo, hi + 1, size=n).astype(np.int32)


def lognormal_lengths(seed: int, n: int, mu: float, sigma: float, lo: int, hi: int) -> np.ndarray:
    z = _rng(seed, _S_SEQLENS).standard_normal(n)
    return np.clip(np.floor(np.exp(mu + sigma * z)), lo, hi).astype(np.int32)


def tiny_decode(seed: int = 0) -> DecodeInputs:
    """B=2, Hq=8, Hk=4, D=64, seq_lens {37, 130}, an 8-page pool.

    The block table is [2, 3]: row 1 uses 3 pages and row 0 uses 1, so five
    distinct ids of a seeded permutation of the 8 pages are placed in it --
    row 0 = (perm[0], perm[4], 0), row 1 = (perm[1], perm[2], perm[3]).
    Row 0's second entry lies past ceil(37/64) = 1 page: it is a stale slot
    that must never be read.
    """
    perm = _rng(seed, _S_PERM).permutation(8).astype(np.int32)
    bt = np.array([[perm[0], perm[4], 0], [perm[1], perm[2], perm[3]]], dtype=np.int32)
    pool_shape = (8, 4, PAGE_SIZE, 64)
    n = int(np.prod(pool_shape))
    return DecodeInputs(
        q=bf16_normal(seed, _S_Q, (2, 8, 64)),
        k_pool=f32_to_bf16_bits(normal_f32(seed, _S_K, n)).reshape(pool_shape),
        v_pool=f32_to_bf16_bits(normal_f32(seed, _S_V, n)).reshape(pool_shape),
        block_table=bt, seq_lens=np.array([37, 130], dtype=np.int32),
        scale=1.0 / 8.0, kv_dtype="bf16")


def gqa_decode(seed: int = 0, batch: int = 64, kv_dtype: str = "bf16") -> DecodeInputs:
    """B=64, Hq=32, Hk=8, D=128, bf16 (or fp16), lengths uniform in [1, 4096]."""
    lens = uniform_lengths(seed, batch, 1, 4096)
    return make_decode(batch, 32, 8, 128, lens, seed, kv_dtype, max_pages=64)


def fp8_long_decode(seed: int = 0, batch: int = 128) -> DecodeInputs:
    """B=128, Hq=64, Hk=8, D=128, e4m3 KV, lengths lognormal(ln 2048, 1) in [64, 16384]."""
    lens = lognormal_lengths(seed, batch, math.log(2048.0), 1.0, 64, 16384)
    return make_decode(batch, 64, 8, 128, lens, seed, "e4m3", max_pages=256)


@dataclass
class PrefillInputs:
    q: np.ndarray             # uint16 [total_q, Hq, Dqk]
    k: np.ndarray             # paged: [P, Hk, 64, Dk]; ragged: [total_k, Hk, Dk]
    v: np.ndarray             # paged: [P, Hk, 64, Dv]; ragged: [total_k, Hk, Dv]
    cu_seqlens_q: np.ndarray  # int32 [B+1]
    cu_seqlens_k: np.ndarray  # int32 [B+1] (kv lengths as running offsets)
    scale: float
    causal: bool = True
    block_table: Optional[np.ndarray] = None   # int32 [B, max_pages] when paged
    k_rope: Optional[np.ndarray] = None        # uint16 [total_k, 1, rope_dim]
    qo_offset: Optional[np.ndarray] = None     # int32 [B] (None: kv_len - q_len)
    dtype: str = "bf16"                         # element type of q, k, v, k_rope: "bf16" | "f16"
    meta: dict = field(default_factory=dict)

    @property
    def batch(self): return len(self.cu_seqlens_q) - 1
    @property
    def num_q_heads(self): return self.q.shape[1]
    @property
    def num_kv_heads(self): return self.k.shape[1]
    @property
    def head_dim_qk(self): return self.q.shape[2]
    @property
    def head_dim_v(self): return self.v.shape[-1]
    @property
    def rope_dim(self): return 0 if self.k_rope is None else self.k_rope.shape[-1]
    @property
    def paged(self): return self.block_table is not None
    @property
    def max_seqlen_q(self): return int(np.max(np.diff(self.cu_seqlens_q))) if self.batch else 0


def make_paged_prefill(q_lens, kv_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                       seed: int = 0, extra_pages: int = 0, qo_offset=None,
                       causal: bool = True, dtype: str = "bf16") -> PrefillInputs:
    q_lens = np.asarray(q_lens, dtype=np.int32)
    kv_lens = np.asarray(kv_lens, dtype=np.int32)
    bt, num_pool = assign_pages(kv_lens, seed, extra_pages)
    total_q = int(q_lens.sum())
    pool_shape = (num_pool, num_kv_heads, PAGE_SIZE, head_dim)
    return PrefillInputs(
        q=normal_16(seed, _S_Q, (total_q, num_q_heads, head_dim), dtype),
        k=normal_16(seed, _S_K, pool_shape, dtype),
        v=normal_16(seed, _S_V, pool_shape, dtype),
        cu_seqlens_q=cu_seqlens(q_lens), cu_seqlens_k=cu_seqlens(kv_lens),
        scale=1.0 / math.sqrt(head_dim), causal=causal, block_table=bt,
        qo_offset=None if qo_offset is None else np.asarray(qo_offset, dtype=np.int32), dtype=dtype)


def chunked_prefill(seed: int = 0, batch: int = 8, q_len: int = 512, max_prefix: int = 8192,
                    heads: int = 32, head_dim: int = 128, dtype: str = "bf16") -> PrefillInputs:
    """q_len new tokens per sequence after a cached prefix uniform in [0, max_prefix]."""
    prefix = _rng(seed, _S_PREFIX).integers(0, max_prefix + 1, size=batch).astype(np.int32)
    q_lens = np.full(batch, q_len, dtype=np.int32)
    p = make_paged_prefill(q_lens, prefix + q_len, heads, heads, head_dim, seed, dtype=dtype)
    p.meta["prefix"] = prefix
    return p


def make_ragged_prefill(lens, num_heads: int, head_dim_qk: int, head_dim_v: int,
                        rope_dim: int = 0, seed: int = 0, num_kv_heads: Optional[int] = None,
                        kv_lens=None, causal: bool = True, qo_offset=None, dtype: str = "bf16") -> PrefillInputs:
    """Ragged q/k/v packed by running offsets; with rope_dim > 0 the MLA layout:
    q [T, H, Dk + rope], k [T, H, Dk], k_rope [T, 1, rope], v [T, H, Dv]."""
    lens = np.asarray(lens, dtype=np.int32)
    kv_lens = lens if kv_lens is None else np.asarray(kv_lens, dtype=np.int32)
    hk = num_heads if num_kv_heads is None else num_kv_heads
    tq, tk = int(lens.sum()), int(kv_lens.sum())
    dk = head_dim_qk - rope_dim
    return PrefillInputs(
        q=normal_16(seed, _S_Q, (tq, num_heads, head_dim_qk), dtype),
        k=normal_16(seed, _S_K, (tk, hk, dk), dtype),
        v=normal_16(seed, _S_V, (tk, hk, head_dim_v), dtype),
        cu_seqlens_q=cu_seqlens(lens), cu_seqlens_k=cu_seqlens(kv_lens),
        scale=1.0 / math.sqrt(head_dim_qk), causal=causal,
        k_rope=normal_16(seed, _S_KROPE, (tk, 1, rope_dim), dtype) if rope_dim else None,
        qo_offset=None if qo_offset is None else np.asarray(qo_offset, dtype=np.int32), dtype=dtype)


def mixed_batch(seed: int = 0) -> PrefillInputs:
    """A serving step's batch: the GQA decode workload's 64 single-token
    sequences (kv lengths uniform in [1, 4096]) followed by the chunked-prefill
    workload's 8 sequences of 512 new tokens after a prefix uniform in [0, 8192];
    Hq=32, Hk=8, D=128, bf16, one paged pool, one ragged query layout."""
    dec = uniform_lengths(seed, 64, 1, 4096)
    prefix = _rng(seed, _S_PREFIX).integers(0, 8193, size=8).astype(np.int32)
    q_lens = np.concatenate([np.ones(64, np.int32), np.full(8, 512, np.int32)])
    kv_lens = np.concatenate([dec, prefix + 512]).astype(np.int32)
    p = make_paged_prefill(q_lens, kv_lens, 32, 8, 128, seed)
    p.meta["num_decode"] = 64
    return p


def mla_prefill(seed: int = 0, batch: int = 8, lo: int = 512, hi: int = 4096,
                heads: int = 128) -> PrefillInputs:
    """8 sequences, lengths uniform in [512, 4096]; q 192 = 128 nope + 64 rope; v 128."""
    lens = uniform_lengths(seed, batch, lo, hi)
    return make_ragged_prefill(lens, heads, 192, 128, rope_dim=64, seed=seed)


@dataclass
class MlaE4m3Inputs:
    """MLA prefill with the per-head parts of q and k in e4m3 plus fp32 scales."""
    q_nope: np.ndarray        # uint8 e4m3 [total_q, Hq, 128]
    q_rope: np.ndarray        # uint16 bf16 [total_q, Hq, 64]
    q_scale: np.ndarray       # float32 [Hq]
    k_nope: np.ndarray        # uint8 e4m3 [total_k, Hk, 128]
    k_scale: np.ndarray       # float32 [Hk]
    k_rope: np.ndarray        # uint16 bf16 [total_k, 1, 64]
    v: np.ndarray             # uint16 bf16 [total_k, Hk, 128]
    cu_seqlens_q: np.ndarray
    cu_seqlens_k: np.ndarray
    scale: float
    causal: bool = True
    qo_offset: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.cu_seqlens_q) - 1

    @property
    def num_q_heads(self) -> int:
        return self.q_nope.shape[1]

    @property
    def num_kv_heads(self) -> int:
        return self.k_nope.shape[1]

    @property
    def max_seqlen_q(self) -> int:
        return int(np.diff(self.cu_seqlens_q).max()) if self.batch else 0

    head_dim_qk = 192
    head_dim_v = 128
    rope_dim = 64
    block_table = None
    paged = False


def _quantise_heads_3d(x: np.ndarray):
    """[T, H, D] float32 -> (e4m3 codes, float32 [H] scales), one scale per head
    (amax / 448, the rule of quantise_per_head)."""
    t, h, d = x.shape
    codes, scales = quantise_per_head(x.reshape(t, h, 1, d))
    return codes.reshape(t, h, d), scales


def make_mla_e4m3(lens, num_heads: int, seed: int = 0, num_kv_heads: Optional[int] = None, kv_lens=None,
                  causal: bool = True, qo_offset=None) -> MlaE4m3Inputs:
    """Ragged MLA prefill with e4m3 q_nope / k_nope: N(0,1) float32 quantised per
    head; q_rope, k_rope and v N(0,1) rounded to bf16; scale 1/sqrt(192)."""
    lens = np.asarray(lens, dtype=np.int32)
    kv_lens = lens if kv_lens is None else np.asarray(kv_lens, dtype=np.int32)
    hk = num_heads if num_kv_heads is None else num_kv_heads
    tq, tk = int(lens.sum()), int(kv_lens.sum())
    qn, qs = _quantise_heads_3d(normal_f32(seed, _S_Q, tq * num_heads * 128).reshape(tq, num_heads, 128))
    kn, ks = _quantise_heads_3d(normal_f32(seed, _S_K, tk * hk * 128).reshape(tk, hk, 128))
    return MlaE4m3Inputs(
        q_nope=qn, q_rope=bf16_normal(seed, _S_QROPE, (tq, num_heads, 64)), q_scale=qs,
        k_nope=kn, k_scale=ks, k_rope=bf16_normal(seed, _S_KROPE, (tk, 1, 64)),
        v=bf16_normal(seed, _S_V, (tk, hk, 128)),
        cu_seqlens_q=cu_seqlens(lens), cu_seqlens_k=cu_seqlens(kv_lens), scale=1.0 / math.sqrt(192.0),
        causal=causal, qo_offset=None if qo_offset is None else np.asarray(qo_offset, dtype=np.int32))


def mla_e4m3_prefill(seed: int = 0, batch: int = 8, lo: int = 512, hi: int = 4096,
                     heads: int = 128) -> MlaE4m3Inputs:
    """The MLA prefill workload's lengths and heads with e4m3 q_nope / k_nope."""
    return make_mla_e4m3(uniform_lengths(seed, batch, lo, hi), heads, seed=seed)


@dataclass
class MlaRopeE4m3Inputs:
    """MLA prefill with the shared rope key in e4m3 plus one fp32 scale per key
    token; q, the per-head k and v in bf16."""
    q: np.ndarray              # uint16 bf16 [total_q, Hq, 192]
    k_nope: np.ndarray         # uint16 bf16 [total_k, Hk, 128]
    v: np.ndarray              # uint16 bf16 [total_k, Hk, 128]
    k_rope: np.ndarray         # uint8 e4m3 [total_k, 1, 64]
    k_rope_scales: np.ndarray  # float32 [total_k]
    cu_seqlens_q: np.ndarray
    cu_seqlens_k: np.ndarray
    scale: float
    causal: bool = True
    qo_offset: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.cu_seqlens_q) - 1

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[1]

    @property
    def num_kv_heads(self) -> int:
        return self.k_nope.shape[1]

    @property
    def max_seqlen_q(self) -> int:
        return int(np.diff(self.cu_seqlens_q).max()) if self.batch else 0

    head_dim_qk = 192
    head_dim_v = 128
    rope_dim = 64
    block_table = None
    paged = False


def quantise_per_row(x: np.ndarray):
    """x float32 [T, D] -> (e4m3 codes [T, D], float32 [T] scales): scale_t =
    amax(|x[t]|) / 448 (1 for an all-zero row), code = e4m3(clamp(float32(x /
    scale_t), -448, 448)), rounded to nearest even (the rule of quantise_per_head,
    one scale per row)."""
    import torch
    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    amax = xt.abs().amax(dim=1) if x.shape[1] else torch.zeros(x.shape[0])
    scales = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    y = (xt / scales.view(-1, 1)).clamp_(-E4M3_MAX, E4M3_MAX)
    return _to_e4m3_bits_fast(y.numpy()).reshape(x.shape), scales.numpy()


def make_mla_rope_e4m3(lens, num_heads: int, seed: int = 0, num_kv_heads: Optional[int] = None, kv_lens=None,
                       causal: bool = True, qo_offset=None) -> MlaRopeE4m3Inputs:
    """Ragged MLA prefill whose rope key is e4m3 with one scale per token: q,
    k_nope and v N(0,1) rounded to bf16, k_rope N(0,1) quantised per token;
    scale 1/sqrt(192)."""
    lens = np.asarray(lens, dtype=np.int32)
    kv_lens = lens if kv_lens is None else np.asarray(kv_lens, dtype=np.int32)
    hk = num_heads if num_kv_heads is None else num_kv_heads
    tq, tk = int(lens.sum()), int(kv_lens.sum())
    codes, scales = quantise_per_row(normal_f32(seed, _S_KROPE, tk * 64).reshape(tk, 64))
    return MlaRopeE4m3Inputs(
        q=bf16_normal_fast(seed, _S_Q, (tq, num_heads, 192)), k_nope=bf16_normal_fast(seed, _S_K, (tk, hk, 128)),
        v=bf16_normal_fast(seed, _S_V, (tk, hk, 128)), k_rope=codes.reshape(tk, 1, 64), k_rope_scales=scales,
        cu_seqlens_q=cu_seqlens(lens), cu_seqlens_k=cu_seqlens(kv_lens), scale=1.0 / math.sqrt(192.0),
        causal=causal, qo_offset=None if qo_offset is None else np.asarray(qo_offset, dtype=np.int32))


def mla_rope_e4m3_prefill(seed: int = 0, batch: int = 8, lo: int = 512, hi: int = 4096,
                          heads: int = 128) -> MlaRopeE4m3Inputs:
    """The MLA prefill workload's lengths and heads with an e4m3 rope key."""
    return make_mla_rope_e4m3(uniform_lengths(seed, batch, lo, hi), heads, seed=seed)


def poison_unused(inp: DecodeInputs, nan_bits: Optional[int] = None) -> DecodeInputs:
    """Fill every pool row that no sequence may read with NaN.

    Rows at or past seq_len in a sequence's last page, and whole pages not
    referenced by any live block-table slot, become NaN (bf16 0x7FC0, e4m3
    0x7F).  A correct kernel never reads them, so its outputs do not change.
    """
    if nan_bits is None:
        nan_bits = 0x7FC0 if inp.kv_dtype == "bf16" else 0x7F
    k = inp.k_pool.copy()
    v = inp.v_pool.copy()
    live = np.zeros((inp.num_pool_pages, PAGE_SIZE), dtype=bool)
    for b, s in enumerate(inp.seq_lens):
        for j in range(pages_for(s)):
            rows = min(PAGE_SIZE, int(s) - j * PAGE_SIZE)
            live[inp.block_table[b, j], :rows] = True
    dead = ~live  # [P, 64]
    k[:, :, :, :][np.broadcast_to(dead[:, None, :, None], k.shape)] = nan_bits
    v[:, :, :, :][np.broadcast_to(dead[:, None, :, None], v.shape)] = nan_bits
    out = DecodeInputs(**{**inp.__dict__})
    out.k_pool, out.v_pool = k, v
    return out


def poison_stale_slots(inp: DecodeInputs, value: int = 2**31 - 1) -> DecodeInputs:
    """Put an out-of-range page id in every block-table slot past ceil(seq_len/64)."""
    bt = inp.block_table.copy()
    for b, s in enumerate(inp.seq_lens):
        bt[b, pages_for(s):] = value
    out = DecodeInputs(**{**inp.__dict__})
    out.block_table = bt
    return out
