"""Guard regions around every buffer a call writes.

The FlashMLA page's paged-cache notes say unused block-table slots are
ignored through seq_lens: nothing outside what a call is given may be
touched.  compute-sanitizer is closed on this machine, so these tests stand in
for its out-of-bounds check on the writes: out, lse, the workspace (and, for
the append, the K/V pools) are carved out of larger device buffers whose
leading and trailing 4 KiB hold a known byte pattern, each call runs at
edge lengths (empty sequences, one key, page and tile boundaries, ragged
tails, split-KV partials), and the guards must come back unchanged.  The
results are checked against the oracle as well, so a write that lands in the
wrong place inside a buffer fails too.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_fwd_gb300 import binding as B
from paged_kv_attention_fwd_gb300 import ops
from paged_kv_attention_fwd_gb300 import workloads as W
from paged_kv_attention_fwd_gb300.build import build

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


class Guarded:
    """`nbytes` of device memory (viewed as `dtype` of `shape`) between two
    GUARD-byte regions filled with PATTERN; the body is filled with `fill`."""

    def __init__(self, shape, dtype, fill=0):
        esize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(shape)) * esize
        self.raw = torch.full((2 * GUARD + self.nbytes,), PATTERN, dtype=torch.uint8, device="cuda")
        self.body = self.raw[GUARD:GUARD + self.nbytes]
        self.body.fill_(fill)
        self.t = self.body.view(dtype).view(shape)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        head, tail = self.raw[:GUARD], self.raw[GUARD + self.nbytes:]
        return bool((head == PATTERN).all().item() and (tail == PATTERN).all().item())


def guarded_copy(src: torch.Tensor) -> Guarded:
    g = Guarded(tuple(src.shape), src.dtype)
    g.t.copy_(src)
    return g


EDGE_LENS = [0, 1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 1000, 4000]


@pytest.mark.parametrize("kv_dtype,forced", [("bf16", 0), ("bf16", 3), ("e4m3", 0), ("e4m3", 5), ("f16", 2)])
def test_decode_writes_stay_inside_out_lse_and_workspace(kv_dtype, forced):
    inp = W.make_decode(len(EDGE_LENS), 16, 4, 128, EDGE_LENS, seed=70, kv_dtype=kv_dtype, extra_pages=2)
    dev = "cuda"
    q = ops.as_f16(inp.q, dev) if kv_dtype == "f16" else ops.as_bf16(inp.q, dev)
    conv = {"bf16": ops.as_bf16, "e4m3": ops.as_e4m3, "f16": ops.as_f16}[kv_dtype]
    kp, vp = conv(inp.k_pool, dev), conv(inp.v_pool, dev)
    ks = torch.from_numpy(inp.k_scale).to(dev) if kv_dtype == "e4m3" else None
    vs = torch.from_numpy(inp.v_scale).to(dev) if kv_dtype == "e4m3" else None
    bt = torch.from_numpy(inp.block_table).to(dev)
    sl = torch.from_numpy(inp.seq_lens).to(dev)
    p = ops.plan_decode(inp.seq_lens, inp.block_table, 16, 4, 128, inp.max_pages, inp.num_pool_pages, kv_dtype,
                        forced_splits=forced)
    if forced:
        assert p.plan.total_splits > inp.batch
    odt = torch.float16 if kv_dtype == "f16" else torch.bfloat16
    out = Guarded((inp.batch, 16, 128), odt)
    lse = Guarded((inp.batch, 16), torch.float32)
    ws = Guarded((p.plan.workspace_bytes,), torch.uint8)
    for fused in (True, False):
        if fused:
            B.pa_decode(p.shapes, p.plan, q, kp, vp, ks, vs, bt, sl, p.meta_dev, inp.scale, out.t, lse.t, ws.t)
        else:
            B.pa_decode_attend(p.shapes, p.plan, q, kp, vp, ks, vs, bt, sl, p.meta_dev, inp.scale, out.t, lse.t,
                               ws.t)
            B.pa_decode_combine(p.shapes, p.plan, p.meta_dev, out.t, lse.t, ws.t)
        assert B.pa_check_status(ws.t) == B.PA_OK
        assert out.intact() and lse.intact() and ws.intact()
    ro, rl = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale, kv_dtype,
                           inp.k_scale, inp.v_scale)
    tol = 5e-2 if kv_dtype == "e4m3" else 1e-2
    assert np.abs(out.t.float().cpu().numpy() - ro).max() <= tol
    got_l = lse.t.cpu().numpy()
    assert np.array_equal(np.isneginf(got_l), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.abs(got_l[fin] - rl[fin]).max() <= 1e-3


@pytest.mark.parametrize("kind", ["paged", "ragged", "mla"])
def test_prefill_writes_stay_inside_out_lse_and_workspace(kind):
    if kind == "paged":
        inp = W.make_paged_prefill([1, 5, 127, 128, 129, 300], [1, 70, 127, 700, 129, 1300], 8, 2, 128, seed=71,
                                   extra_pages=2)
    elif kind == "ragged":
        inp = W.make_ragged_prefill([1, 2, 127, 128, 129, 255, 256, 257, 513], 4, 128, 128, seed=72,
                                    num_kv_heads=2)
    else:
        inp = W.make_ragged_prefill([1, 63, 129, 256, 300], 8, 192, 128, rope_dim=64, seed=73)
    dev = "cuda"
    tq = int(inp.cu_seqlens_q[-1])
    sh = ops.prefill_shapes(inp.batch, inp.num_q_heads, inp.num_kv_heads, inp.head_dim_qk, inp.head_dim_v,
                            inp.rope_dim, inp.max_seqlen_q, tq, int(inp.cu_seqlens_k[-1]),
                            max_pages=inp.block_table.shape[1] if inp.paged else 0,
                            num_pool_pages=inp.k.shape[0] if inp.paged else 0)
    out = Guarded((tq, inp.num_q_heads, 128), torch.bfloat16)
    lse = Guarded((tq, inp.num_q_heads), torch.float32)
    ws = Guarded((B.pa_prefill_workspace_size(sh),), torch.uint8)
    kr = ops.as_bf16(inp.k_rope, dev) if inp.k_rope is not None else None
    bt = torch.from_numpy(inp.block_table).to(dev) if inp.paged else None
    for _ in range(2):  # the second call reuses the workspace's work counters
        B.pa_prefill(sh, ops.as_bf16(inp.q, dev), ops.as_bf16(inp.k, dev), ops.as_bf16(inp.v, dev), kr,
                     torch.from_numpy(inp.cu_seqlens_q).to(dev), torch.from_numpy(inp.cu_seqlens_k).to(dev), bt,
                     None, True, inp.scale, out.t, lse.t, ws.t)
        assert B.pa_check_status(ws.t) == B.PA_OK
        assert out.intact() and lse.intact() and ws.intact()
    ro, rl = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                            block_table=inp.block_table, k_rope=inp.k_rope)
    assert np.abs(out.t.float().cpu().numpy() - ro).max() <= 1e-2
    assert np.abs(lse.t.cpu().numpy() - rl).max() <= 1e-3


def test_mixed_writes_stay_inside_out_lse_and_workspace():
    q_lens, kv_lens = [1, 1, 1, 40, 300, 1, 128], [700, 1, 3000, 40, 1300, 65, 2000]
    inp = W.make_paged_prefill(q_lens, kv_lens, 8, 2, 128, seed=74, extra_pages=2)
    dev = "cuda"
    kl = np.diff(inp.cu_seqlens_k).astype(np.int32)
    sh = B.pa_mixed_shapes(batch=inp.batch, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=64,
                           max_pages_per_seq=inp.block_table.shape[1], num_pool_pages=inp.k.shape[0],
                           kv_dtype=B.PA_KV_BF16, num_sms=ops.num_sms(), ctas_per_sm=0, forced_splits=0)
    meta, plan = B.pa_get_mixed_plan(inp.cu_seqlens_q, kl, inp.block_table, sh)
    tq = int(inp.cu_seqlens_q[-1])
    out = Guarded((tq, 8, 128), torch.bfloat16)
    lse = Guarded((tq, 8), torch.float32)
    ws = Guarded((plan.workspace_bytes,), torch.uint8)
    B.pa_mixed(sh, plan, ops.as_bf16(inp.q, dev), ops.as_bf16(inp.k, dev), ops.as_bf16(inp.v, dev),
               torch.from_numpy(inp.block_table).to(dev), torch.from_numpy(inp.cu_seqlens_q).to(dev),
               torch.from_numpy(inp.cu_seqlens_k).to(dev), torch.from_numpy(kl).to(dev),
               torch.from_numpy(meta).to(dev), inp.scale, out.t, lse.t, ws.t)
    torch.cuda.synchronize()
    assert out.intact() and lse.intact() and ws.intact()
    ro, rl = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                            block_table=inp.block_table)
    assert np.abs(out.t.float().cpu().numpy() - ro).max() <= 1e-2
    assert np.abs(lse.t.cpu().numpy() - rl).max() <= 1e-3


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_append_writes_stay_inside_the_pools(kv_dtype):
    prior = np.array([0, 63, 64, 130, 1000], np.int32)
    new = np.array([5, 1, 70, 200, 64], np.int32)
    base = W.make_decode(len(prior), 4, 4, 128, prior + new, seed=75, kv_dtype=kv_dtype, extra_pages=3)
    dev = "cuda"
    kn = W.normal_16(75, 90, (int(new.sum()), 4, 128), "bf16")
    vn = W.normal_16(75, 91, (int(new.sum()), 4, 128), "bf16")
    conv = ops.as_e4m3 if kv_dtype == "e4m3" else ops.as_bf16
    kp, vp = guarded_copy(conv(base.k_pool, dev)), guarded_copy(conv(base.v_pool, dev))
    ws = Guarded((B.PA_STATUS_BYTES,), torch.uint8)
    sh = B.pa_append_shapes(batch=len(prior), num_kv_heads=4, head_dim=128, page_size=64,
                            max_pages_per_seq=base.block_table.shape[1], num_pool_pages=base.num_pool_pages,
                            total_new=int(new.sum()),
                            kv_dtype=B.PA_KV_FP8_E4M3 if kv_dtype == "e4m3" else B.PA_KV_BF16)
    ks = torch.from_numpy(base.k_scale).to(dev) if kv_dtype == "e4m3" else None
    vs = torch.from_numpy(base.v_scale).to(dev) if kv_dtype == "e4m3" else None
    B.pa_append_kv(sh, ops.as_bf16(kn, dev), ops.as_bf16(vn, dev), torch.from_numpy(W.cu_seqlens(new)).to(dev),
                   torch.from_numpy(prior).to(dev), torch.from_numpy(base.block_table).to(dev), kp.t, vp.t, ks, vs,
                   ws.t)
    assert B.pa_check_status(ws.t) == B.PA_OK
    assert kp.intact() and vp.intact() and ws.intact()
    k_ref, v_ref = oracle.append_kv(kn, vn, W.cu_seqlens(new), prior, base.block_table, base.k_pool, base.v_pool,
                                    base.k_scale, base.v_scale)
    raw = torch.uint8 if kv_dtype == "e4m3" else torch.int16
    assert np.array_equal(kp.t.view(raw).cpu().numpy().view(k_ref.dtype), k_ref)
    assert np.array_equal(vp.t.view(raw).cpu().numpy().view(v_ref.dtype), v_ref)
