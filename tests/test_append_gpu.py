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


def test_append_then_decode_steps_without_sync():
    """Decode steps as a serving loop issues them: every round appends one new
    token per sequence, then decodes over the grown cache, all on one stream
    with no host synchronisation between the launches.  The decode may start
    its prologue while the append is still running (the append lets its
    dependents launch as soon as it starts), so a decode that read pages
    before the append completed would see the stale tokens the pool was
    filled with.  Every round must match the oracle on the pool as it stood
    after that round's append."""
    rounds, hq, hk, d = 4, 16, 4, 128
    prior = np.array([0, 63, 64, 300, 1000, 5, 129, 2047], np.int32)
    nb = len(prior)
    base = W.make_decode(nb, hq, hk, d, prior + rounds, seed=52, kv_dtype="bf16", extra_pages=3)
    dev = "cuda"
    kp, vp = ops.as_bf16(base.k_pool, dev), ops.as_bf16(base.v_pool, dev)
    bt = torch.from_numpy(base.block_table).to(dev)
    cu = torch.from_numpy(np.arange(nb + 1, dtype=np.int32)).to(dev)
    kn = [W.bf16_normal(52, 100 + r, (nb, hk, d)) for r in range(rounds)]
    vn = [W.bf16_normal(52, 110 + r, (nb, hk, d)) for r in range(rounds)]
    qs = [W.bf16_normal(52, 120 + r, (nb, hq, d)) for r in range(rounds)]
    kn_d, vn_d, q_d = ([ops.as_bf16(x, dev) for x in xs] for xs in (kn, vn, qs))
    start_d = [torch.from_numpy(prior + r).to(dev) for r in range(rounds)]
    lens_d = [torch.from_numpy(prior + r + 1).to(dev) for r in range(rounds)]
    plans = [ops.plan_decode(prior + r + 1, base.block_table, hq, hk, d, base.max_pages, base.num_pool_pages)
             for r in range(rounds)]
    sh = B.pa_append_shapes(batch=nb, num_kv_heads=hk, head_dim=d, page_size=64,
                            max_pages_per_seq=base.block_table.shape[1], num_pool_pages=base.num_pool_pages,
                            total_new=nb, kv_dtype=B.PA_KV_BF16)
    ws = torch.zeros(B.PA_STATUS_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    outs = []
    for r in range(rounds):
        B.pa_append_kv(sh, kn_d[r], vn_d[r], cu, start_d[r], bt, kp, vp, None, None, ws)
        outs.append(ops.decode(plans[r], q_d[r], kp, vp, bt, lens_d[r], base.scale))
    torch.cuda.synchronize()
    assert B.pa_check_status(ws) == B.PA_OK
    k_ref, v_ref = base.k_pool, base.v_pool
    cu_h = np.arange(nb + 1, dtype=np.int32)
    for r in range(rounds):
        assert B.pa_check_status(plans[r].workspace) == B.PA_OK
        k_ref, v_ref = oracle.append_kv(kn[r], vn[r], cu_h, prior + r, base.block_table, k_ref, v_ref)
        ro, rl = oracle.decode(qs[r], k_ref, v_ref, base.block_table, prior + r + 1, base.scale)
        out, lse = outs[r][0].float().cpu().numpy(), outs[r][1].cpu().numpy()
        err = np.abs(out - ro)
        assert err.max() <= 1e-2 and err.mean() <= 1e-3, f"round {r}: max abs err {err.max():.3g}"
        assert np.abs(lse - rl).max() <= 1e-3, f"round {r}"


def test_append_then_chunked_prefill_without_sync():
    """The chunked-prefill flow on one stream with no host synchronisation:
    the prefill reads the pages the append has just written (the pool holds
    stale random tokens at those positions before the append)."""
    prefix = np.array([0, 70, 500, 64], np.int32)
    qlen = np.array([40, 129, 256, 300], np.int32)
    base, _, _, kn, vn = case("bf16", hk=4, prior=prefix, new=qlen, seed=53)
    dev = "cuda"
    kp, vp = ops.as_bf16(base.k_pool, dev), ops.as_bf16(base.v_pool, dev)
    bt = torch.from_numpy(base.block_table).to(dev)
    q = W.bf16_normal(53, 92, (int(qlen.sum()), 8, 128))
    q_d, kn_d, vn_d = ops.as_bf16(q, dev), ops.as_bf16(kn, dev), ops.as_bf16(vn, dev)
    cu_new = torch.from_numpy(W.cu_seqlens(qlen)).to(dev)
    start = torch.from_numpy(prefix).to(dev)
    cu_k = torch.from_numpy(W.cu_seqlens(prefix + qlen)).to(dev)
    sh_app = B.pa_append_shapes(batch=len(prefix), num_kv_heads=4, head_dim=128, page_size=64,
                                max_pages_per_seq=base.block_table.shape[1], num_pool_pages=base.num_pool_pages,
                                total_new=int(qlen.sum()), kv_dtype=B.PA_KV_BF16)
    sh = ops.prefill_shapes(len(prefix), 8, 4, 128, 128, 0, int(qlen.max()), int(qlen.sum()),
                            int((prefix + qlen).sum()), max_pages=base.max_pages, num_pool_pages=base.num_pool_pages)
    ws = torch.zeros(B.PA_STATUS_BYTES, dtype=torch.uint8, device=dev)
    pws = torch.zeros(B.pa_prefill_workspace_size(sh), dtype=torch.uint8, device=dev)
    out = torch.empty((int(qlen.sum()), 8, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((int(qlen.sum()), 8), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    # the append and the prefill launches are adjacent in the stream
    B.pa_append_kv(sh_app, kn_d, vn_d, cu_new, start, bt, kp, vp, None, None, ws)
    ops.prefill(sh, q_d, kp, vp, cu_new, cu_k, base.scale, True, block_table=bt, out=out, lse=lse, workspace=pws)
    torch.cuda.synchronize()
    assert B.pa_check_status(ws) == B.PA_OK and B.pa_check_status(pws) == B.PA_OK
    k_ref, v_ref = oracle.append_kv(kn, vn, W.cu_seqlens(qlen), prefix, base.block_table, base.k_pool, base.v_pool)
    ro, rl = oracle.prefill(q, k_ref, v_ref, W.cu_seqlens(qlen), W.cu_seqlens(prefix + qlen), base.scale, True,
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
