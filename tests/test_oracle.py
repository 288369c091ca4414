"""Pins for the CPU oracle: closed forms, invariants, page-printed fixtures and
library routines (torch CPU float64), chosen so that a dropped term, a wrong
index, sign or grouping in the oracle fails at least one of them."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_fwd_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return np.array(rows)


def t_bf16(bits):
    """bf16 bit patterns -> float64 through torch's own bfloat16 type."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float64)


def t_e4m3(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.float8_e4m3fn).to(torch.float64)


# ---------------------------------------------------------------- element decoders

def test_bf16_decoder_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = t_bf16(codes).numpy()
    got = oracle.bf16_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_decoder_all_codes():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.float16).to(torch.float64).numpy()
    got = oracle.f16_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], ref[~nan])


def t_f16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16).to(torch.float64)


def test_e4m3_decoder_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = t_e4m3(codes).numpy()
    got = oracle.e4m3_to_f64(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_generator_encoders_match_torch():
    x = W.normal_f32(3, 99, 20000) * np.float32(40.0)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.f32_to_bf16_bits(x), ref)
    xc = np.clip(x, -448, 448)
    ref8 = torch.from_numpy(xc).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(W.f32_to_e4m3_bits(xc), ref8)
    # saturation beyond the largest finite value
    assert W.f32_to_e4m3_bits(np.array([1e6, -1e6])).tolist() == [0x7E, 0xFE]


# ---------------------------------------------------------------- library cross-check

def _gather_dense(pool, bt_row, n):
    """[Hk, n, D] keys of one sequence via torch indexing (a route independent of the oracle)."""
    pages = torch.as_tensor(bt_row[: (n + 63) // 64], dtype=torch.long)
    blk = pool[pages]                          # [np, Hk, 64, D]
    return blk.permute(1, 0, 2, 3).reshape(pool.shape[1], -1, pool.shape[-1])[:, :n]


def _sdpa(q, k, v, scale, mask=None):
    """torch float64 attention; q [H, Lq, D], k/v [H, Lk, *]; returns out, lse."""
    out = torch.nn.functional.scaled_dot_product_attention(
        q[None], k[None], v[None], attn_mask=mask, scale=scale)[0]
    s = (q @ k.transpose(-1, -2)) * scale
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    return out, torch.logsumexp(s, dim=-1)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3", "f16"])
def test_decode_matches_torch_sdpa(kv_dtype):
    inp = W.make_decode(3, 8, 2, 64, [1, 65, 200], seed=5, kv_dtype=kv_dtype, extra_pages=3)
    out, lse = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens,
                             inp.scale, kv_dtype, inp.k_scale, inp.v_scale)
    dec = {"bf16": t_bf16, "e4m3": t_e4m3, "f16": t_f16}[kv_dtype]
    kp, vp = dec(inp.k_pool), dec(inp.v_pool)
    if kv_dtype == "e4m3":
        kp = kp * torch.as_tensor(inp.k_scale, dtype=torch.float64)[None, :, None, None]
        vp = vp * torch.as_tensor(inp.v_scale, dtype=torch.float64)[None, :, None, None]
    q = t_f16(inp.q) if kv_dtype == "f16" else t_bf16(inp.q)
    G = inp.num_q_heads // inp.num_kv_heads
    for b, n in enumerate(inp.seq_lens):
        k = _gather_dense(kp, inp.block_table[b], int(n)).repeat_interleave(G, 0)
        v = _gather_dense(vp, inp.block_table[b], int(n)).repeat_interleave(G, 0)
        ro, rl = _sdpa(q[b][:, None, :], k, v, inp.scale)
        np.testing.assert_allclose(out[b], ro[:, 0].numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl[:, 0].numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_paged_prefill_matches_torch_sdpa(dtype):
    inp = W.make_paged_prefill([5, 70, 1], [40, 200, 64], 4, 2, 64, seed=9, extra_pages=2, dtype=dtype)
    out, lse = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale,
                              True, block_table=inp.block_table, dtype=dtype)
    dec = t_f16 if dtype == "f16" else t_bf16
    kp, vp, q = dec(inp.k), dec(inp.v), dec(inp.q)
    for b in range(inp.batch):
        q0, q1 = inp.cu_seqlens_q[b], inp.cu_seqlens_q[b + 1]
        n = int(inp.cu_seqlens_k[b + 1] - inp.cu_seqlens_k[b])
        lq = q1 - q0
        k = _gather_dense(kp, inp.block_table[b], n).repeat_interleave(2, 0)
        v = _gather_dense(vp, inp.block_table[b], n).repeat_interleave(2, 0)
        mask = torch.ones(lq, n, dtype=torch.bool).tril(diagonal=n - lq)
        ro, rl = _sdpa(q[q0:q1].transpose(0, 1), k, v, inp.scale, mask)
        np.testing.assert_allclose(out[q0:q1], ro.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[q0:q1], rl.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_mla_ragged_matches_concatenated_keys():
    """MLA reduces exactly to standard attention with K = [k_nope[h], k_rope]."""
    inp = W.make_ragged_prefill([9, 130], 4, 48, 32, rope_dim=16, seed=2)
    out, lse = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale,
                              True, k_rope=inp.k_rope)
    q, k, v, kr = t_bf16(inp.q), t_bf16(inp.k), t_bf16(inp.v), t_bf16(inp.k_rope)
    for b in range(inp.batch):
        a, e = inp.cu_seqlens_q[b], inp.cu_seqlens_q[b + 1]
        L = e - a
        kk = torch.cat([k[a:e], kr[a:e].expand(L, 4, 16)], dim=-1).transpose(0, 1)
        ro, rl = _sdpa(q[a:e].transpose(0, 1), kk, v[a:e].transpose(0, 1), inp.scale,
                       torch.ones(L, L, dtype=torch.bool).tril())
        np.testing.assert_allclose(out[a:e], ro.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[a:e], rl.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_prefix_zero_is_textbook_causal():
    inp = W.make_ragged_prefill([33], 2, 32, 32, seed=4)
    out, lse = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True)
    q, k, v = (t_bf16(x).transpose(0, 1) for x in (inp.q, inp.k, inp.v))
    ref = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True,
                                                           scale=inp.scale)[0]
    np.testing.assert_allclose(out, ref.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def _dec(bits):
    return t_bf16(bits).numpy()


def test_single_key_gives_v0_and_score():
    inp = W.make_decode(2, 4, 2, 64, [1, 1], seed=11)
    out, lse = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale)
    for b in range(2):
        page = inp.block_table[b, 0]
        for h in range(4):
            kv = h // 2
            v0 = _dec(inp.v_pool[page, kv, 0])
            k0 = _dec(inp.k_pool[page, kv, 0])
            assert np.array_equal(out[b, h], v0)
            assert lse[b, h] == pytest.approx(inp.scale * float(np.dot(_dec(inp.q[b, h]), k0)), rel=1e-13)


def test_zero_query_gives_mean_of_v_and_log_n():
    inp = W.make_decode(2, 2, 1, 64, [100, 7], seed=12)
    inp.q[:] = 0
    out, lse = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale)
    vp = _dec(inp.v_pool)
    for b, n in enumerate(inp.seq_lens):
        rows = np.concatenate([vp[inp.block_table[b, j], 0] for j in range((n + 63) // 64)])[:n]
        np.testing.assert_allclose(out[b, 0], rows.mean(0), rtol=0, atol=1e-14)
        assert lse[b, 0] == pytest.approx(math.log(n), abs=1e-14)


def test_constant_v_gives_v():
    inp = W.make_decode(3, 4, 4, 64, [5, 64, 129], seed=13)
    c = W.f32_to_bf16_bits(np.linspace(-2, 2, 64, dtype=np.float32))
    inp.v_pool[:] = c
    out, _ = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale)
    np.testing.assert_allclose(out, np.broadcast_to(_dec(c), out.shape), rtol=0, atol=1e-14)


def test_output_in_convex_hull_of_values():
    inp = W.make_decode(2, 4, 2, 64, [90, 3], seed=14)
    out, _ = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale)
    vp = _dec(inp.v_pool)
    for b, n in enumerate(inp.seq_lens):
        for h in range(4):
            rows = np.concatenate([vp[inp.block_table[b, j], h // 2] for j in range((n + 63) // 64)])[:n]
            assert np.all(out[b, h] <= rows.max(0) + 1e-12) and np.all(out[b, h] >= rows.min(0) - 1e-12)


def test_empty_key_set():
    inp = W.make_decode(2, 2, 1, 64, [0, 3], seed=15)
    out, lse = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0])) and np.all(np.isfinite(lse[1]))


# ---------------------------------------------------------------- page-printed fixtures

def test_gqa_grouping_matches_page_diagram():
    """V of kv head g is the constant g; then out of q head h is exactly its kv head."""
    table = _golden("gqa_map_hq8_hk4.txt")
    inp = W.make_decode(1, 8, 4, 64, [77], seed=16)
    for g in range(4):
        inp.v_pool[:, g] = W.f32_to_bf16_bits(np.float32([g]))[0]
    out, _ = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale)
    for qh, kvh in table:
        np.testing.assert_allclose(out[0, qh], kvh, rtol=1e-14, atol=0)
        others = [g for g in range(4) if g != kvh]
        assert all(np.all(np.abs(out[0, qh] - g) > 0.5) for g in others)


def test_token_to_page_mapping_matches_page_diagram():
    """With q = 0 the output is the mean of the visible V rows; marking the rows of
    one physical page with 1 reveals exactly which tokens that page serves."""
    table = _golden("token_page_map.txt")
    n = 192
    inp = W.make_decode(1, 1, 1, 64, [n], seed=17, extra_pages=2)
    inp.q[:] = 0
    one = W.f32_to_bf16_bits(np.float32([1.0]))[0]
    for first, last, col in table:
        inp.v_pool[:] = 0
        inp.v_pool[inp.block_table[0, col]] = one
        out, _ = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale)
        np.testing.assert_allclose(out[0, 0], (last - first + 1) / n, atol=1e-15)
        # shortening the sequence to end inside this range keeps only its first tokens
        m = first + 10
        out2, _ = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, np.array([m], np.int32),
                                inp.scale)
        np.testing.assert_allclose(out2[0, 0], 10 / m, atol=1e-15)


# ---------------------------------------------------------------- invariants

def test_page_permutation_invariance_exact():
    inp = W.make_decode(3, 4, 2, 64, [64, 150, 20], seed=18, extra_pages=4)
    out, lse = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale)
    perm = np.random.default_rng(0).permutation(inp.num_pool_pages)
    inv = np.argsort(perm)
    k2 = inp.k_pool[perm]     # new page i holds old page perm[i]
    v2 = inp.v_pool[perm]
    bt2 = inv[inp.block_table].astype(np.int32)
    out2, lse2 = oracle.decode(inp.q, k2, v2, bt2, inp.seq_lens, inp.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_poisoned_unused_rows_and_slots_change_nothing(kv_dtype):
    inp = W.make_decode(3, 4, 2, 64, [37, 130, 64], seed=19, kv_dtype=kv_dtype, extra_pages=3,
                        max_pages=5)
    args = (inp.scale, kv_dtype, inp.k_scale, inp.v_scale)
    out, lse = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, *args)
    p = W.poison_stale_slots(W.poison_unused(inp))
    out2, lse2 = oracle.decode(p.q, p.k_pool, p.v_pool, p.block_table, p.seq_lens, *args)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    assert np.all(np.isfinite(out2))


def test_decode_equals_prefill_with_one_query_row():
    inp = W.make_decode(3, 4, 2, 64, [1, 100, 257], seed=20)
    out, lse = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale)
    cu_q = W.cu_seqlens(np.ones(3, np.int32))
    cu_k = W.cu_seqlens(inp.seq_lens)
    out2, lse2 = oracle.prefill(inp.q, inp.k_pool, inp.v_pool, cu_q, cu_k, inp.scale, True,
                                block_table=inp.block_table)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-15)


def test_chunk_row_equals_decode_at_its_length():
    """Row i of a causal chunk with offset o sees exactly keys 0 .. o + i."""
    inp = W.make_paged_prefill([20], [150], 2, 2, 64, seed=21)
    out, lse = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale,
                              True, block_table=inp.block_table)
    off = 150 - 20
    for i in (0, 7, 19):
        lens = np.array([off + i + 1], np.int32)
        o, l = oracle.decode(inp.q[i:i + 1], inp.k, inp.v, inp.block_table, lens, inp.scale)
        np.testing.assert_allclose(out[i], o[0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[i], l[0], rtol=0, atol=1e-15)


def test_explicit_qo_offset_and_non_causal():
    inp = W.make_paged_prefill([8, 8], [64, 100], 2, 1, 64, seed=22)
    default = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                             block_table=inp.block_table)
    explicit = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                              block_table=inp.block_table, qo_offset=np.array([56, 92], np.int32))
    assert np.array_equal(default[0], explicit[0])
    # an offset past the end sees every key: same as non-causal
    wide = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                          block_table=inp.block_table, qo_offset=np.array([1000, 1000], np.int32))
    nc = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, False,
                        block_table=inp.block_table)
    assert np.array_equal(wide[0], nc[0])
    # a negative offset hides keys; row i sees min(kv_len, max(i + 1 + off, 0)) keys
    neg = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                         block_table=inp.block_table, qo_offset=np.array([-3, 0], np.int32))
    assert np.all(np.isneginf(neg[1][:3, :])) and np.all(np.isfinite(neg[1][3:8]))


def test_paged_prefill_refuses_keys_past_the_block_table():
    """A paged segment's keys are addressed through its block-table row (the
    FlashMLA paged-cache diagram: page block_table[b, j // 64], row j % 64); a
    kv_len above max_pages * 64 has no page for its last keys, and the oracle
    refuses it instead of reading the next row of the table."""
    inp = W.make_paged_prefill([4, 4], [64, 100], 2, 1, 64, seed=25)
    assert inp.block_table.shape[1] == 2
    cu_k = inp.cu_seqlens_k.copy()
    cu_k[1:] += 200  # sequence 0 now claims 264 keys, more than 2 pages hold
    with pytest.raises(ValueError):
        oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, cu_k, inp.scale, True, block_table=inp.block_table)
    # at exactly max_pages * 64 keys the call is valid
    cu_ok = np.array([0, 128, 228], np.int32)
    bt = inp.block_table.copy()
    oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, cu_ok, inp.scale, True, block_table=bt)


def test_ragged_equals_separate_calls():
    inp = W.make_ragged_prefill([5, 40, 17], 4, 32, 32, seed=23, num_kv_heads=2)
    out, lse = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True)
    for b in range(3):
        a, e = inp.cu_seqlens_q[b], inp.cu_seqlens_q[b + 1]
        cu = np.array([0, e - a], np.int32)
        o, l = oracle.prefill(inp.q[a:e], inp.k[a:e], inp.v[a:e], cu, cu, inp.scale, True)
        assert np.array_equal(o, out[a:e]) and np.array_equal(l, lse[a:e])


def test_row_sampling_matches_full():
    inp = W.make_ragged_prefill([30, 45], 4, 32, 32, seed=24, rope_dim=0)
    out, lse = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True)
    rows = np.array([0, 5, 4 * 30 + 3, 4 * 74 + 3], np.int64)
    o, l = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                          rows=rows)
    flat_o = out.reshape(-1, 32)
    assert np.array_equal(o, flat_o[rows]) and np.array_equal(l, lse.reshape(-1)[rows])


def test_fp8_scales_fold_into_scores_and_values():
    """Dequantisation multiplies each element by its head's scale: doubling the
    K scale doubles every score (same as doubling the softmax scale) and the
    V scale multiplies the output."""
    inp = W.make_decode(2, 4, 2, 64, [70, 9], seed=25, kv_dtype="e4m3")
    base = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale,
                         "e4m3", inp.k_scale, inp.v_scale)
    o2 = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, 2 * inp.scale,
                       "e4m3", inp.k_scale, 3 * inp.v_scale.astype(np.float64))
    o3 = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale,
                       "e4m3", 2 * inp.k_scale.astype(np.float64), inp.v_scale)
    np.testing.assert_allclose(o2[0], 3 * o3[0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(o2[1], o3[1], rtol=1e-12)
    assert not np.allclose(base[0], o3[0])


def test_generator_fast_paths_equal_reference_encoders():
    x = W.normal_f32(7, 98, 50000) * np.float32(3.0)
    assert np.array_equal(W._to_bf16_bits_fast(x), W.f32_to_bf16_bits(x))
    pool = x[: 4 * 2 * 64 * 48].reshape(4, 2, 64, 48)
    fast, s1 = W.quantise_per_head(pool, fast=True)
    ref, s2 = W.quantise_per_head(pool, fast=False)
    assert np.array_equal(fast, ref) and np.array_equal(s1, s2)
    # every head uses its full range: the largest magnitude encodes to +-448
    dec = oracle.e4m3_to_f64(fast.reshape(-1)).reshape(fast.shape)
    assert np.allclose(np.abs(dec).max(axis=(0, 2, 3)), 448.0)


# ---------------------------------------------------------------- paged KV append

def test_e4m3_encoder_matches_torch():
    x = np.concatenate([W.normal_f32(8, 97, 40000) * np.float32(60.0),
                        np.float32([0.0, -0.0, 448.0, 460.0, 1e-9, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -6 * 0.9375])])
    xc = np.clip(x, -448, 448)
    ref = torch.from_numpy(xc).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_from_f32(xc)
    assert np.array_equal(got, ref)
    assert oracle.e4m3_from_f32(np.float32([1e6, -1e6])).tolist() == [0x7E, 0xFE]  # saturates


def _append_case(kv_dtype, seed=40):
    hk, d = 2, 64
    prior = np.array([0, 63, 64, 130], np.int32)   # cached tokens before the append
    new = np.array([5, 1, 70, 200], np.int32)
    base = W.make_decode(4, 4, hk, d, prior + new, seed=seed, kv_dtype=kv_dtype, extra_pages=2)
    kn = W.bf16_normal(seed, 90, (int(new.sum()), hk, d))
    vn = W.bf16_normal(seed, 91, (int(new.sum()), hk, d))
    return base, prior, new, kn, vn


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_append_then_decode_sees_the_new_tokens(kv_dtype):
    """Appending at position prior_b and decoding over prior_b + new_b keys equals
    attention over keys gathered from the old pool (first prior_b) followed by
    the new rows -- the token -> page mapping of the page diagram."""
    base, prior, new, kn, vn = _append_case(kv_dtype)
    cu = W.cu_seqlens(new)
    kp, vp = oracle.append_kv(kn, vn, cu, prior, base.block_table, base.k_pool, base.v_pool,
                              base.k_scale, base.v_scale)
    # untouched rows are unchanged; written rows hold exactly the (quantised) new values
    enc = (lambda x, s: x) if kv_dtype == "bf16" else (
        lambda x, s: oracle.e4m3_from_f32(t_bf16(x).numpy().astype(np.float32) / s[None, :, None]))
    changed = 0
    for b in range(4):
        for i in range(new[b]):
            p = prior[b] + i
            pg, r = base.block_table[b, p // 64], p % 64
            row_k = enc(kn[cu[b] + i][None], base.k_scale)[0] if kv_dtype == "e4m3" else kn[cu[b] + i]
            assert np.array_equal(kp[pg, :, r], row_k)
            changed += 1
    diff = np.any(kp != base.k_pool, axis=(1, 3))  # [P, 64] rows touched
    assert diff.sum() <= changed * 1  # nothing else written
    out, lse = oracle.decode(base.q, kp, vp, base.block_table, prior + new, base.scale, kv_dtype,
                             base.k_scale, base.v_scale)
    # reference: keys from the old pool for the prior tokens, then the new rows
    dec = t_bf16 if kv_dtype == "bf16" else t_e4m3
    for b in range(4):
        pages = base.block_table[b, : (prior[b] + new[b] + 63) // 64]
        kk = dec(kp)[pages].permute(1, 0, 2, 3).reshape(2, -1, 64)[:, : prior[b] + new[b]]
        vv = dec(vp)[pages].permute(1, 0, 2, 3).reshape(2, -1, 64)[:, : prior[b] + new[b]]
        if kv_dtype == "e4m3":
            kk = kk * torch.as_tensor(base.k_scale, dtype=torch.float64)[:, None, None]
            vv = vv * torch.as_tensor(base.v_scale, dtype=torch.float64)[:, None, None]
        ro, rl = _sdpa(t_bf16(base.q[b])[:, None, :], kk.repeat_interleave(2, 0), vv.repeat_interleave(2, 0),
                       base.scale)
        np.testing.assert_allclose(out[b], ro[:, 0].numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl[:, 0].numpy(), rtol=1e-12, atol=1e-12)
    # the bf16 append is an exact copy: decoding only the new tokens of a sequence
    # whose cache was empty (b = 0) sees exactly the appended values
    if kv_dtype == "bf16":
        np.testing.assert_array_equal(kp[base.block_table[0, 0], :, :5], np.transpose(kn[:5], (1, 0, 2)))


# ---------------------------------------------------------------- fp8 MLA prefill

def _mla_e4m3_small(seed=7, heads=4, hk=None):
    return W.make_mla_e4m3([9, 130, 1], heads, seed=seed, num_kv_heads=hk)


def test_mla_e4m3_with_power_of_two_scales_equals_the_bf16_mla_oracle():
    """e4m3 values times powers of two are exactly representable in bf16: the fp8
    MLA oracle must then reproduce the (separately pinned) bf16 MLA oracle bit for
    bit on the same values -- a dropped scale, a swapped operand or a wrong head
    index breaks the equality."""
    inp = _mla_e4m3_small(heads=4, hk=2)
    rng = np.random.default_rng(0)
    inp.q_scale = np.exp2(rng.integers(-9, -3, size=4)).astype(np.float32)
    inp.k_scale = np.exp2(rng.integers(-9, -3, size=2)).astype(np.float32)
    lut = t_e4m3(np.arange(256, dtype=np.uint8)).numpy()
    qn = lut[inp.q_nope] * inp.q_scale[None, :, None]
    kn = lut[inp.k_nope] * inp.k_scale[None, :, None]
    q16 = np.concatenate([W.f32_to_bf16_bits(qn.astype(np.float32)), inp.q_rope], axis=-1)
    k16 = W.f32_to_bf16_bits(kn.astype(np.float32))
    assert np.array_equal(t_bf16(k16).numpy(), kn)  # the re-encoding is exact
    ref_out, ref_lse = oracle.prefill(q16, k16, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                                      k_rope=inp.k_rope)
    out, lse = oracle.prefill_mla_e4m3(inp.q_nope, inp.q_rope, inp.q_scale, inp.k_nope, inp.k_scale, inp.v,
                                       inp.k_rope, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)


def test_mla_e4m3_matches_torch_sdpa_with_general_scales():
    inp = _mla_e4m3_small(seed=8)
    out, lse = oracle.prefill_mla_e4m3(inp.q_nope, inp.q_rope, inp.q_scale, inp.k_nope, inp.k_scale, inp.v,
                                       inp.k_rope, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale)
    qs = torch.from_numpy(inp.q_scale.astype(np.float64))[None, :, None]
    ks = torch.from_numpy(inp.k_scale.astype(np.float64))[None, :, None]
    q = torch.cat([t_e4m3(inp.q_nope) * qs, t_bf16(inp.q_rope)], dim=-1)
    k = t_e4m3(inp.k_nope) * ks
    v, kr = t_bf16(inp.v), t_bf16(inp.k_rope)
    for b in range(inp.batch):
        a, e = inp.cu_seqlens_q[b], inp.cu_seqlens_q[b + 1]
        L = e - a
        kk = torch.cat([k[a:e], kr[a:e].expand(L, 4, 64)], dim=-1).transpose(0, 1)
        ro, rl = _sdpa(q[a:e].transpose(0, 1), kk, v[a:e].transpose(0, 1), inp.scale,
                       torch.ones(L, L, dtype=torch.bool).tril())
        np.testing.assert_allclose(out[a:e], ro.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[a:e], rl.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_mla_e4m3_scale_moves_between_q_and_k():
    """Only q_scale * k_scale matters: multiplying one by c and dividing the
    other by c leaves the result unchanged (up to double rounding)."""
    inp = _mla_e4m3_small(seed=9)
    args = (inp.v, inp.k_rope, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale)
    o1, l1 = oracle.prefill_mla_e4m3(inp.q_nope, inp.q_rope, inp.q_scale, inp.k_nope, inp.k_scale, *args)
    o2, l2 = oracle.prefill_mla_e4m3(inp.q_nope, inp.q_rope, (inp.q_scale * 3).astype(np.float32), inp.k_nope,
                                     (inp.k_scale.astype(np.float64) / 3).astype(np.float32), *args)
    # float32 scales: (3 q)(k / 3) differs from q k by at most a few float32 ulps
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-5)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-5)
    # and the rope term is not scaled: doubling q_scale changes the result
    o3, _ = oracle.prefill_mla_e4m3(inp.q_nope, inp.q_rope, (inp.q_scale * 2).astype(np.float32), inp.k_nope,
                                    inp.k_scale, *args)
    assert np.abs(o3 - o1).max() > 1e-3


# ---------------------------------------------------------------- MLA with an e4m3 rope key

def _mla_rope_e4m3_small(seed=11, heads=4, hk=None):
    return W.make_mla_rope_e4m3([9, 130, 1], heads, seed=seed, num_kv_heads=hk)


def _rope_e4m3_oracle(inp, **kw):
    return oracle.prefill_mla_rope_e4m3(inp.q, inp.k_nope, inp.v, inp.k_rope, inp.k_rope_scales, inp.cu_seqlens_q,
                                        inp.cu_seqlens_k, inp.scale, **kw)


def test_mla_rope_e4m3_with_power_of_two_scales_equals_the_bf16_mla_oracle():
    """An e4m3 code times a power of two (or zero) is exactly a bf16 value, so with
    such per-token scales the oracle must reproduce the (separately pinned) bf16
    MLA oracle bit for bit on the decoded rope key -- a scale applied per head or
    per query row instead of per key token, or to the whole score instead of the
    rope term, breaks the equality."""
    inp = _mla_rope_e4m3_small(hk=2)
    rng = np.random.default_rng(1)
    tk = inp.k_rope.shape[0]
    sc = np.exp2(rng.integers(-9, 2, size=tk)).astype(np.float32)
    sc[5] = 0.0  # a token whose rope term vanishes
    inp.k_rope_scales = sc
    kr = t_e4m3(inp.k_rope).numpy() * sc[:, None, None]
    kr16 = W.f32_to_bf16_bits(kr.astype(np.float32))
    assert np.array_equal(t_bf16(kr16).numpy(), kr)  # the re-encoding is exact
    ref_out, ref_lse = oracle.prefill(inp.q, inp.k_nope, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                                      k_rope=kr16)
    out, lse = _rope_e4m3_oracle(inp)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)


def test_mla_rope_e4m3_matches_torch_sdpa_with_general_scales():
    inp = _mla_rope_e4m3_small(seed=12)
    out, lse = _rope_e4m3_oracle(inp)
    kr = t_e4m3(inp.k_rope) * torch.from_numpy(inp.k_rope_scales.astype(np.float64))[:, None, None]
    q, k, v = t_bf16(inp.q), t_bf16(inp.k_nope), t_bf16(inp.v)
    for b in range(inp.batch):
        a, e = inp.cu_seqlens_q[b], inp.cu_seqlens_q[b + 1]
        L = e - a
        kk = torch.cat([k[a:e], kr[a:e].expand(L, 4, 64)], dim=-1).transpose(0, 1)
        ro, rl = _sdpa(q[a:e].transpose(0, 1), kk, v[a:e].transpose(0, 1), inp.scale,
                       torch.ones(L, L, dtype=torch.bool).tril())
        np.testing.assert_allclose(out[a:e], ro.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[a:e], rl.transpose(0, 1).numpy(), rtol=1e-12, atol=1e-12)


def test_mla_rope_e4m3_scale_multiplies_only_that_tokens_rope_term():
    """Scaling token t's rope scale by c equals scaling its rope codes' values by
    c: with c = 2 (exact) the result equals the oracle on codes re-encoded at
    twice the value, and the change reaches only rows that can see token t."""
    inp = _mla_rope_e4m3_small(seed=13)
    o1, l1 = _rope_e4m3_oracle(inp)
    t = int(inp.cu_seqlens_k[-1]) - 1  # the last token: only the one-row third sequence sees it
    sc = inp.k_rope_scales.copy()
    sc[t] *= 2
    inp2 = W.MlaRopeE4m3Inputs(**{**inp.__dict__, "k_rope_scales": sc})
    o2, l2 = _rope_e4m3_oracle(inp2)
    first = int(inp.cu_seqlens_q[2])
    assert np.array_equal(o1[:first], o2[:first]) and np.array_equal(l1[:first], l2[:first])
    assert np.abs(l2[first:] - l1[first:]).max() > 1e-6
