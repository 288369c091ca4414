"""Device-side scheduling on the GPU: pa_get_metadata_device must write the
oracle's snake-dealt schedule bit for bit, pa_decode must give the same
outputs with it as with the host schedule, and a CUDA graph captured once
(schedule + decode) must give the oracle's results when replayed with new
lengths in the same device buffer."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import scheduler as S
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


def shapes(batch, hq, hk, max_pages, pool, forced=0, kv=B.PA_KV_BF16, sms=None):
    return B.pa_decode_shapes(batch=batch, num_q_heads=hq, num_kv_heads=hk, head_dim=128, page_size=64,
                              max_pages_per_seq=max_pages, num_pool_pages=pool, kv_dtype=kv,
                              num_sms=sms or ops.num_sms(), ctas_per_sm=0, forced_splits=forced)


def device_meta(sh, lens):
    plan = B.pa_get_static_plan(sh)
    meta = torch.full((plan.meta_ints,), -7, dtype=torch.int32, device="cuda")
    B.pa_get_metadata_device(sh, plan, torch.from_numpy(np.asarray(lens, np.int32)).cuda(), meta)
    torch.cuda.synchronize()
    return plan, meta


@pytest.mark.parametrize("case", ["uniform", "lognormal", "forced", "edges", "single", "mid", "large", "wide"])
def test_device_schedule_bit_exact(case):
    cases = ["uniform", "lognormal", "forced", "edges", "single", "large", "wide", "mid"]
    rng = np.random.default_rng(100 + cases.index(case))
    if case == "uniform":
        lens, hk, forced, mp = rng.integers(1, 4097, 64), 8, 0, 64
    elif case == "lognormal":
        lens, hk, forced, mp = np.clip(np.floor(np.exp(math.log(2048) + rng.standard_normal(128))), 64, 16384), 8, 0, 256
    elif case == "forced":
        lens, hk, forced, mp = rng.integers(0, 3000, 40), 4, 7, 64
    elif case == "edges":
        lens, hk, forced, mp = np.array([0, 1, 63, 64, 65, 128, 129, 4096, 0, 5000]), 2, 0, 100
    elif case == "single":
        lens, hk, forced, mp = np.array([1]), 1, 0, 1
    elif case == "mid":  # ~1000 splits: the 256-thread schedule
        lens, hk, forced, mp = rng.integers(0, 3001, 900), 4, 0, 64
    elif case == "large":  # ~14700 items
        lens, hk, forced, mp = rng.integers(0, 2001, 1800), 8, 0, 32
    else:  # one KV head: as many splits as items, the sort's 16 keys per thread
        lens, hk, forced, mp = rng.integers(0, 4097, 8192), 1, 2, 64
    lens = lens.astype(np.int32)
    sh = shapes(len(lens), hk * 2, hk, mp, 10 ** 6, forced)
    plan, meta = device_meta(sh, lens)
    ref = S.schedule(lens.tolist(), hk, sh.num_sms, 1, forced, dealing="snake")
    got = meta.cpu().numpy()
    assert got[: len(ref)].tolist() == ref
    assert len(ref) <= plan.meta_ints and S.unpack(ref)["total_splits"] <= plan.total_splits


def _decode_inputs(seed=70, B=24):
    lens = W.uniform_lengths(seed, B, 1, 3000)
    return W.make_decode(B, 32, 8, 128, lens, seed=seed, max_pages=48)


def test_decode_with_device_schedule_equals_host_schedule():
    inp = _decode_inputs()
    dev = "cuda"
    q, kp, vp = ops.as_bf16(inp.q, dev), ops.as_bf16(inp.k_pool, dev), ops.as_bf16(inp.v_pool, dev)
    bt, sl = torch.from_numpy(inp.block_table).to(dev), torch.from_numpy(inp.seq_lens).to(dev)
    host = ops.plan_decode(inp.seq_lens, inp.block_table, 32, 8, 128, inp.max_pages, inp.num_pool_pages)
    o1, l1 = ops.decode(host, q, kp, vp, bt, sl, inp.scale)
    sh = shapes(inp.batch, 32, 8, inp.max_pages, inp.num_pool_pages)
    plan, meta = device_meta(sh, inp.seq_lens)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    o2 = torch.empty_like(o1)
    l2 = torch.empty_like(l1)
    B.pa_decode(sh, plan, q, kp, vp, None, None, bt, sl, meta, inp.scale, o2, l2, ws)
    assert B.pa_check_status(ws) == B.PA_OK and B.pa_check_status(host.workspace) == B.PA_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)  # same splits, same merge order


def test_cuda_graph_replay_with_new_lengths():
    seed, Bsz = 71, 24
    cap_lens = np.full(Bsz, 3000, np.int32)
    inp = W.make_decode(Bsz, 32, 8, 128, cap_lens, seed=seed, max_pages=48)  # pages for the longest case
    dev = "cuda"
    q, kp, vp = ops.as_bf16(inp.q, dev), ops.as_bf16(inp.k_pool, dev), ops.as_bf16(inp.v_pool, dev)
    bt = torch.from_numpy(inp.block_table).to(dev)
    sl = torch.from_numpy(cap_lens.copy()).to(dev)
    sh = shapes(Bsz, 32, 8, inp.max_pages, inp.num_pool_pages)
    plan = B.pa_get_static_plan(sh)
    meta = torch.zeros(plan.meta_ints, dtype=torch.int32, device=dev)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((Bsz, 32, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Bsz, 32), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()

    def step():
        B.pa_get_metadata_device(sh, plan, sl, meta, stream=s)
        B.pa_decode(sh, plan, q, kp, vp, None, None, bt, sl, meta, inp.scale, out, lse, ws, stream=s)

    with torch.cuda.stream(s):
        step()  # eager once: first launches configure the kernels
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    rng = np.random.default_rng(seed)
    for trial in range(3):
        lens = rng.integers(0 if trial else 1, 3001, Bsz).astype(np.int32)
        sl.copy_(torch.from_numpy(lens))
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, lens, inp.scale)
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        err = np.abs(o - ref_out)
        assert err.max() <= 1e-2 and err.mean() <= 1e-3
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isneginf(l), np.isneginf(ref_lse))
        assert np.abs(l[fin] - ref_lse[fin]).max() <= 1e-3
    assert B.pa_check_status(ws) == B.PA_OK


def test_cuda_graph_replay_full_size():
    """The graph-replayed decode at the bench's full size (B=64, Hq=32, Hk=8,
    D=128, lengths U[1,4096]): the scheduler and the decode captured once,
    replayed with the workload's lengths and then with shorter random ones;
    every sequence against the oracle."""
    inp = W.gqa_decode(0)
    dev = "cuda"
    q, kp, vp = ops.as_bf16(inp.q, dev), ops.as_bf16(inp.k_pool, dev), ops.as_bf16(inp.v_pool, dev)
    bt = torch.from_numpy(inp.block_table).to(dev)
    sl = torch.from_numpy(inp.seq_lens.copy()).to(dev)
    sh = shapes(inp.batch, 32, 8, inp.max_pages, inp.num_pool_pages)
    plan = B.pa_get_static_plan(sh)
    meta = torch.zeros(plan.meta_ints, dtype=torch.int32, device=dev)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((inp.batch, 32, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((inp.batch, 32), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()

    def step():
        B.pa_get_metadata_device(sh, plan, sl, meta, stream=s)
        B.pa_decode(sh, plan, q, kp, vp, None, None, bt, sl, meta, inp.scale, out, lse, ws, stream=s)

    with torch.cuda.stream(s):
        step()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    rng = np.random.default_rng(72)
    for lens in (inp.seq_lens, np.minimum(inp.seq_lens, rng.integers(1, 4097, inp.batch)).astype(np.int32)):
        sl.copy_(torch.from_numpy(np.ascontiguousarray(lens)))
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, lens, inp.scale)
        err = np.abs(out.float().cpu().numpy() - ref_out)
        assert err.max() <= 1e-2 and err.mean() <= 1e-3, f"max abs err {err.max():.3g}"
        assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 1e-3
    assert B.pa_check_status(ws) == B.PA_OK
