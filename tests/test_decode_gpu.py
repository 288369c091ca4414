"""Decode parity on the GPU: libpa (through the C ABI) against the fp64 oracle
on the same seeded inputs.  Tolerances: bf16 out max-abs 1e-2 and mean-abs
1e-3, e4m3-KV out max-abs 5e-2, lse abs 1e-3; metadata bit-exact."""
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

from .parity import abs_values, assert_close_16, scale_16_bits

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-3), "e4m3": (5e-2, 5e-3), "f16": (1e-2, 1e-3)}
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()
    torch.cuda.init()


def to_dev(inp: W.DecodeInputs, dev="cuda"):
    q = ops.as_f16(inp.q, dev) if inp.kv_dtype == "f16" else ops.as_bf16(inp.q, dev)
    conv = {"bf16": ops.as_bf16, "e4m3": ops.as_e4m3, "f16": ops.as_f16}[inp.kv_dtype]
    kp, vp = conv(inp.k_pool, dev), conv(inp.v_pool, dev)
    bt = torch.from_numpy(np.ascontiguousarray(inp.block_table)).to(dev)
    sl = torch.from_numpy(np.ascontiguousarray(inp.seq_lens)).to(dev)
    ks = vs = None
    if inp.kv_dtype == "e4m3":
        ks = torch.from_numpy(inp.k_scale).to(dev)
        vs = torch.from_numpy(inp.v_scale).to(dev)
    return q, kp, vp, bt, sl, ks, vs


def run(inp: W.DecodeInputs, forced=0, check_host_table=True, **kw):
    q, kp, vp, bt, sl, ks, vs = to_dev(inp)
    p = ops.plan_decode(inp.seq_lens, inp.block_table if check_host_table else None, inp.num_q_heads,
                        inp.num_kv_heads, inp.head_dim, inp.max_pages, inp.num_pool_pages, inp.kv_dtype,
                        forced_splits=forced, **kw)
    out, lse = ops.decode(p, q, kp, vp, bt, sl, inp.scale, ks, vs)
    st = B.pa_check_status(p.workspace)
    return out.float().cpu().numpy(), lse.cpu().numpy(), st, p


def reference(inp: W.DecodeInputs):
    return oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale,
                         inp.kv_dtype, inp.k_scale, inp.v_scale)


def assert_close(out, lse, ref_out, ref_lse, kv_dtype):
    mx, mean = TOL[kv_dtype]
    err = np.abs(out - ref_out)
    assert np.all(np.isfinite(out))
    assert err.max() <= mx, f"max abs err {err.max():.3g}"
    assert err.mean() <= mean, f"mean abs err {err.mean():.3g}"
    neg = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), neg)
    if (~neg).any():
        lerr = np.abs(lse[~neg] - ref_lse[~neg])
        assert lerr.max() <= LSE_TOL, f"lse err {lerr.max():.3g}"


def test_tiny_paged_decode():
    inp = W.tiny_decode(0)
    out, lse, st, p = run(inp)
    assert st == B.PA_OK
    assert out.shape == (2, 8, 64) and lse.shape == (2, 8)
    assert p.meta.tolist() == S.schedule(inp.seq_lens.tolist(), 4, ops.num_sms(), 1)
    ref_out, ref_lse = reference(inp)
    assert_close(out, lse, ref_out, ref_lse, "bf16")


def test_gqa_decode_full_size():
    inp = W.gqa_decode(0)
    out, lse, st, p = run(inp)
    assert st == B.PA_OK
    assert p.plan.total_splits > inp.batch  # the auto rule splits the longer sequences
    ref_out, ref_lse = reference(inp)
    assert_close(out, lse, ref_out, ref_lse, "bf16")


@pytest.mark.parametrize("forced", [1, 2, 7, 0])
def test_split_count_does_not_change_result(forced):
    inp = W.make_decode(8, 32, 8, 128, [1, 64, 65, 700, 1500, 2049, 3000, 129], seed=3)
    out, lse, st, p = run(inp, forced=forced)
    assert st == B.PA_OK
    ref_out, ref_lse = reference(inp)
    assert_close(out, lse, ref_out, ref_lse, "bf16")
    base_out, base_lse, _, _ = run(inp, forced=1)
    assert np.abs(out - base_out).max() <= 1e-2 and np.abs(lse - base_lse).max() <= 1e-4


@pytest.mark.parametrize("hq,hk,d", [(8, 8, 128), (16, 8, 128), (64, 4, 128), (8, 4, 64), (16, 1, 64),
                                     (32, 2, 128), (24, 8, 128), (40, 8, 128), (96, 8, 64)])
def test_group_sizes_and_edge_lengths(hq, hk, d):
    lens = [0, 1, 2, 63, 64, 65, 127, 128, 129, 191, 255, 256, 257, 1000]
    inp = W.make_decode(len(lens), hq, hk, d, lens, seed=hq + hk + d, extra_pages=2)
    out, lse, st, _ = run(inp)
    assert st == B.PA_OK
    ref_out, ref_lse = reference(inp)
    assert_close(out, lse, ref_out, ref_lse, "bf16")
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))


@pytest.mark.parametrize("forced", [0, 3])
def test_poisoned_rows_pages_and_stale_slots(forced):
    inp = W.make_decode(6, 16, 4, 128, [37, 130, 64, 1, 700, 255], seed=4, extra_pages=5, max_pages=16)
    clean = run(inp, forced=forced)
    p = W.poison_stale_slots(W.poison_unused(inp))
    dirty = run(p, forced=forced, check_host_table=False)
    assert dirty[2] == B.PA_OK
    assert np.all(np.isfinite(dirty[0]))
    assert np.array_equal(clean[0], dirty[0]) and np.array_equal(clean[1], dirty[1])
    ref_out, ref_lse = reference(inp)
    assert_close(dirty[0], dirty[1], ref_out, ref_lse, "bf16")


def test_deterministic_bitwise():
    inp = W.make_decode(16, 32, 8, 128, W.uniform_lengths(9, 16, 1, 3000), seed=9)
    a = run(inp)
    b = run(inp)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fp8_kv_decode():
    lens = W.lognormal_lengths(5, 24, math.log(700.0), 1.0, 64, 4000)
    inp = W.make_decode(24, 64, 8, 128, lens, seed=5, kv_dtype="e4m3")
    out, lse, st, p = run(inp)
    assert st == B.PA_OK
    ref_out, ref_lse = reference(inp)
    assert_close(out, lse, ref_out, ref_lse, "e4m3")


# e4m3 at D = 128: groups of <= 4 and <= 8 heads run two softmax warpgroups,
# larger groups one; non-power-of-two groups pad the softmax heads
@pytest.mark.parametrize("hq,hk,d", [(8, 4, 64), (16, 16, 128), (24, 8, 128), (40, 8, 128), (64, 8, 128),
                                     (128, 8, 128), (12, 1, 128)])
def test_fp8_edges(hq, hk, d):
    lens = [0, 1, 63, 64, 65, 129, 300]
    inp = W.make_decode(len(lens), hq, hk, d, lens, seed=6, kv_dtype="e4m3", extra_pages=3)
    p = W.poison_unused(inp)
    out, lse, st, _ = run(p)
    assert st == B.PA_OK
    ref_out, ref_lse = reference(inp)
    assert_close(out, lse, ref_out, ref_lse, "e4m3")


def test_fp8_long_context_full_size():
    """The full long-context e4m3 workload (B=128, Hq=64, Hk=8, lognormal
    lengths up to 16384, split-KV with the fused merge): every output of every
    sequence against the oracle."""
    inp = W.fp8_long_decode(0)
    out, lse, st, p = run(inp)
    assert st == B.PA_OK
    assert p.plan.total_splits > inp.batch
    ref_out, ref_lse = reference(inp)
    assert_close(out, lse, ref_out, ref_lse, "e4m3")


def test_device_bounds_are_reported_not_faulted():
    inp = W.make_decode(2, 8, 4, 128, [100, 200], seed=7)
    bad = W.DecodeInputs(**{**inp.__dict__})
    bad.block_table = inp.block_table.copy()
    bad.block_table[1, 2] = inp.num_pool_pages + 5  # live slot (200 keys -> 4 pages)
    out, lse, st, _ = run(bad, check_host_table=False)
    assert st == B.PA_ERR_DEVICE_BOUNDS
    # the context is still usable and a clean call still succeeds
    out2, lse2, st2, _ = run(inp)
    assert st2 == B.PA_OK
    ref_out, ref_lse = reference(inp)
    assert_close(out2, lse2, ref_out, ref_lse, "bf16")


def test_bounded_wait_times_out_cleanly():
    ws = torch.zeros(B.PA_STATUS_BYTES, dtype=torch.uint8, device="cuda")
    B.pa_debug_wait_timeout(ws, 20_000_000)  # 20 ms on a barrier nothing arrives on
    assert B.pa_check_status(ws) == B.PA_ERR_TIMEOUT
    assert B.pa_check_status(ws) == B.PA_OK  # cleared by the read
    inp = W.tiny_decode(0)
    out, lse, st, _ = run(inp)
    assert st == B.PA_OK


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_fused_merge_matches_two_kernel_form(kv_dtype):
    """pa_decode merges split partials inside its kernel; pa_decode_attend +
    pa_decode_combine do it in a second kernel.  Same results, and the fused
    form leaves its arrival counters at zero for the next call."""
    inp = W.make_decode(12, 32, 8, 128, W.uniform_lengths(13, 12, 1, 4096), seed=13, kv_dtype=kv_dtype)
    q, kp, vp, bt, sl, ks, vs = to_dev(inp)
    p = ops.plan_decode(inp.seq_lens, inp.block_table, 32, 8, 128, inp.max_pages, inp.num_pool_pages, kv_dtype,
                        forced_splits=5)
    assert p.plan.total_splits > inp.batch
    for _ in range(2):  # twice: the counters must have been reset by the first call
        o1, l1 = ops.decode(p, q, kp, vp, bt, sl, inp.scale, ks, vs)
        assert B.pa_check_status(p.workspace) == B.PA_OK
        o2 = torch.empty_like(o1)
        l2 = torch.empty_like(l1)
        B.pa_decode_attend(p.shapes, p.plan, q, kp, vp, ks, vs, bt, sl, p.meta_dev, inp.scale, o2, l2, p.workspace)
        B.pa_decode_combine(p.shapes, p.plan, p.meta_dev, o2, l2, p.workspace)
        assert B.pa_check_status(p.workspace) == B.PA_OK
        assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
        assert (l1 - l2).abs().max().item() <= 1e-5
    ref_out, ref_lse = reference(inp)
    assert_close(o1.float().cpu().numpy(), l1.cpu().numpy(), ref_out, ref_lse, kv_dtype)



@pytest.mark.parametrize("hq,hk,d", [(32, 8, 128), (8, 4, 64), (16, 1, 128)])
def test_fp16_decode(hq, hk, d):
    """fp16 query, pools and output (the three share one type)."""
    lens = [0, 1, 63, 64, 65, 200, 1000, 3000]
    inp = W.make_decode(len(lens), hq, hk, d, lens, seed=80 + hq, kv_dtype="f16", extra_pages=2)
    out, lse, st, p = run(inp)
    assert st == B.PA_OK
    ref_out, ref_lse = reference(inp)
    assert_close(out, lse, ref_out, ref_lse, "f16")


def test_max_batch_host_and_device_plans():
    """8192 sequences, the most the device scheduler takes, lengths U[0, 300]
    (empty, one-page and multi-page sequences mixed), Hq=4, Hk=1, D=64: the
    host plan and the device-written plan both against the oracle."""
    bsz = 8192
    lens = np.random.default_rng(91).integers(0, 301, bsz).astype(np.int32)
    inp = W.make_decode(bsz, 4, 1, 64, lens, seed=91)
    ref_out, ref_lse = reference(inp)
    out, lse, st, p = run(inp)
    assert st == B.PA_OK
    assert_close(out, lse, ref_out, ref_lse, "bf16")
    q, kp, vp, bt, sl, _, _ = to_dev(inp)
    sh = p.shapes
    plan = B.pa_get_static_plan(sh)
    meta = torch.zeros(plan.meta_ints, dtype=torch.int32, device="cuda")
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    o2 = torch.empty((bsz, 4, 64), dtype=torch.bfloat16, device="cuda")
    l2 = torch.empty((bsz, 4), dtype=torch.float32, device="cuda")
    B.pa_get_metadata_device(sh, plan, sl, meta)
    B.pa_decode(sh, plan, q, kp, vp, None, None, bt, sl, meta, inp.scale, o2, l2, ws)
    assert B.pa_check_status(ws) == B.PA_OK
    assert_close(o2.float().cpu().numpy(), l2.cpu().numpy(), ref_out, ref_lse, "bf16")


@pytest.mark.parametrize("kv_dtype", ["bf16", "f16"])
def test_large_outputs_under_the_ulp_rule(kv_dtype):
    """Values 16x larger and queries 16x larger (both exact power-of-two
    scalings of the seeded inputs): outputs averaged from values of magnitude
    up to ~70 by a peaked softmax, where the 1e-2 bar is below the format's
    own rounding; checked under the rule of tests/parity.py (bound 2^-m times
    the weighted mean |v|, which the oracle gives on |V|)."""
    lens = [1, 63, 200, 700, 1500, 2500, 3000, 4000]
    inp = W.make_decode(len(lens), 16, 4, 128, lens, seed=41, kv_dtype=kv_dtype)
    big = W.DecodeInputs(**{**inp.__dict__})
    big.q = scale_16_bits(inp.q, 16.0, kv_dtype)
    big.v_pool = scale_16_bits(inp.v_pool, 16.0, kv_dtype)
    out, lse, st, _ = run(big)
    assert st == B.PA_OK
    ref_out, ref_lse = reference(big)
    absv = W.DecodeInputs(**{**big.__dict__})
    absv.v_pool = abs_values(big.v_pool)
    abs_mean, _ = reference(absv)  # softmax-weighted mean of |v| per output element
    assert np.abs(ref_out).max() >= 8  # the regime this test is about
    assert_close_16(out, lse, ref_out, ref_lse, abs_mean, kv_dtype)
