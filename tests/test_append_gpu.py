"""Paged KV append on the GPU: pa_append_kv (through the C ABI) writes new
tokens into their pages; the pools must match the oracle's bit for bit (bf16
copy, e4m3 nearest-even quantisation), and a chunked prefill right after the
append must match the oracle on the appended pool."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_fwd_gb300 import binding as B
from paged_kv_attention_fwd_gb300 import ops
from paged_kv_attention_fwd_gb300 import workloads as W
from paged_kv_attention_fwd_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


def case(kv_dtype, hk=4, d=128, prior=(0, 63, 64, 130, 1000), new=(5, 1, 70, 200, 64), seed=50):
    prior = np.array(prior, np.int32)
    new = np.array(new, np.int32)
    base = W.make_decode(len(prior), hk, hk, d, prior + new, seed=seed, kv_dtype=kv_dtype, extra_pages=3)
    src = "f16" if kv_dtype == "f16" else "bf16"
    kn = W.normal_16(seed, 90, (int(new.sum()), hk, d), src)
    vn = W.normal_16(seed, 91, (int(new.sum()), hk, d), src)
    return base, prior, new, kn, vn


def gpu_append(base, prior, new, kn, vn, block_table=None):
    dev = "cuda"
    conv = {"bf16": ops.as_bf16, "e4m3": ops.as_e4m3, "f16": ops.as_f16}[base.kv_dtype]
    kp, vp = conv(base.k_pool, dev), conv(base.v_pool, dev)
    bt = base.block_table if block_table is None else block_table
    sh = B.pa_append_shapes(batch=len(prior), num_kv_heads=base.num_kv_heads, head_dim=base.head_dim, page_size=64,
                            max_pages_per_seq=bt.shape[1], num_pool_pages=base.num_pool_pages,
                            total_new=int(new.sum()),
                            kv_dtype={"bf16": B.PA_KV_BF16, "e4m3": B.PA_KV_FP8_E4M3, "f16": B.PA_KV_FP16}[base.kv_dtype])
    ks = torch.from_numpy(base.k_scale).to(dev) if base.k_scale is not None else None
    vs = torch.from_numpy(base.v_scale).to(dev) if base.v_scale is not None else None
    ws = torch.zeros(B.PA_STATUS_BYTES, dtype=torch.uint8, device=dev)
    src = ops.as_f16 if base.kv_dtype == "f16" else ops.as_bf16
    B.pa_append_kv(sh, src(kn, dev), src(vn, dev), torch.from_numpy(W.cu_seqlens(new)).to(dev),
                   torch.from_numpy(prior).to(dev), torch.from_numpy(bt).to(dev), kp, vp, ks, vs, ws)
    st = B.pa_check_status(ws)
    raw = torch.uint8 if base.kv_dtype == "e4m3" else torch.int16
    k_out = kp.view(raw).cpu().numpy().view(base.k_pool.dtype)
    v_out = vp.view(raw).cpu().numpy().view(base.v_pool.dtype)
    return k_out, v_out, st


@pytest.mark.parametrize("kv_dtype,d,hk", [("bf16", 128, 4), ("bf16", 64, 4), ("e4m3", 128, 4), ("e4m3", 64, 4),
                                          ("f16", 128, 4), ("bf16", 128, 3), ("bf16", 64, 5), ("e4m3", 128, 9),
                                          ("bf16", 128, 1)])
def test_append_bit_exact(kv_dtype, d, hk):
    # a warp moves the rows of up to 4 KV heads: head counts that are not a
    # multiple of 4 leave a partial last group
    base, prior, new, kn, vn = case(kv_dtype, d=d, hk=hk)
    k_gpu, v_gpu, st = gpu_append(base, prior, new, kn, vn)
    assert st == B.PA_OK
    k_ref, v_ref = oracle.append_kv(kn, vn, W.cu_seqlens(new), prior, base.block_table, base.k_pool, base.v_pool,
                                    base.k_scale, base.v_scale)
    assert np.array_equal(k_gpu, k_ref) and np.array_equal(v_gpu, v_ref)
    assert not np.array_equal(k_ref, base.k_pool)  # something was written


def test_append_then_chunked_prefill():
    """The chunked-prefill flow: append the chunk's K/V at kv positions
    prefix .. prefix+q_len-1, then attend causally over the whole cache."""
    prefix = np.array([0, 70, 500], np.int32)
    qlen = np.array([40, 129, 256], np.int32)
    base, _, _, kn, vn = case("bf16", hk=4, prior=prefix, new=qlen, seed=51)
    k_gpu, v_gpu, st = gpu_append(base, prefix, qlen, kn, vn)
    assert st == B.PA_OK
    q = W.bf16_normal(51, 92, (int(qlen.sum()), 4, 128))
    inp = W.PrefillInputs(q=q, k=k_gpu, v=v_gpu, cu_seqlens_q=W.cu_seqlens(qlen),
                          cu_seqlens_k=W.cu_seqlens(prefix + qlen), scale=base.scale, causal=True,
                          block_table=base.block_table)
    dev = "cuda"
    sh = ops.prefill_shapes(3, 4, 4, 128, 128, 0, int(qlen.max()), int(qlen.sum()), int((prefix + qlen).sum()),
                            max_pages=base.max_pages, num_pool_pages=base.num_pool_pages)
    out, lse, ws = ops.prefill(sh, ops.as_bf16(q, dev), ops.as_bf16(k_gpu, dev), ops.as_bf16(v_gpu, dev),
                               torch.from_numpy(inp.cu_seqlens_q).to(dev), torch.from_numpy(inp.cu_seqlens_k).to(dev),
                               base.scale, True, block_table=torch.from_numpy(base.block_table).to(dev))
    assert B.pa_check_status(ws) == B.PA_OK
    k_ref, v_ref = oracle.append_kv(kn, vn, W.cu_seqlens(qlen), prefix, base.block_table, base.k_pool, base.v_pool)
    ro, rl = oracle.prefill(q, k_ref, v_ref, inp.cu_seqlens_q, inp.cu_seqlens_k, base.scale, True,
                            block_table=base.block_table)
    err = np.abs(out.float().cpu().numpy() - ro)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3


def test_append_out_of_range_is_reported():
    base, prior, new, kn, vn = case("bf16")
    bt = base.block_table.copy()
    p = prior[2] + new[2] - 1                # last new token of sequence 2
    bt[2, p // 64] = base.num_pool_pages + 7  # its page id is out of the pool
    k_gpu, v_gpu, st = gpu_append(base, prior, new, kn, vn, block_table=bt)
    assert st == B.PA_ERR_DEVICE_BOUNDS
    # every other token was written exactly as the oracle writes it
    new_ok = new.copy()
    k_ref, _ = oracle.append_kv(kn, vn, W.cu_seqlens(new), prior, base.block_table, base.k_pool, base.v_pool)
    page = base.block_table[2, p // 64]
    rows_bad = [(prior[2] + i) % 64 for i in range(new[2]) if (prior[2] + i) // 64 == p // 64]
    mask = np.ones(k_ref.shape[:3], bool)
    mask[page, :, rows_bad] = False
    assert np.array_equal(k_gpu[mask], k_ref[mask])
    assert np.array_equal(k_gpu[page][:, rows_bad], base.k_pool[page][:, rows_bad])  # untouched
