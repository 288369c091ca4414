"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (a host framework that owns all device memory through its own
pool, a loop that cannot pay for an allocation's synchronisation) get one
entry point that uses the library's fixed 16 MiB scratch array instead of a
caller workspace.  These tests call it through the C ABI and check that its
output matches pa_decode's and the fp64 oracle's within the decode
tolerances, on calls made one after another (the scratch keeps the previous
call's contents); that the device status word comes back through
status_host, clean or with a recorded fault; that host-side checks run
before anything is enqueued; and that a plan needing more scratch than the
fixed size is refused with a clear error.
This file is collected last on purpose.
"""
import math

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


def _device_inputs(inp):
    dev = "cuda"
    conv = ops.as_bf16 if inp.kv_dtype == "bf16" else ops.as_e4m3
    ks = torch.from_numpy(inp.k_scale).to(dev) if inp.k_scale is not None else None
    vs = torch.from_numpy(inp.v_scale).to(dev) if inp.v_scale is not None else None
    return (ops.as_bf16(inp.q, dev), conv(inp.k_pool, dev), conv(inp.v_pool, dev), ks, vs,
            torch.from_numpy(inp.block_table).to(dev), torch.from_numpy(inp.seq_lens).to(dev))


def _close(out, lse, ref_out, ref_lse, max_tol, mean_tol):
    o, r = out.float().cpu().numpy(), ref_out.float().cpu().numpy()
    err = np.abs(o - r)
    assert np.all(np.isfinite(o)) and err.max() <= max_tol and err.mean() <= mean_tol
    l, rl = lse.cpu().numpy(), ref_lse.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    assert np.abs(l[fin] - rl[fin]).max() <= 1e-3


def _check_against_pa_decode(inp, calls, max_tol, mean_tol):
    q, kp, vp, ks, vs, bt, sl = _device_inputs(inp)
    p = ops.plan_decode(inp.seq_lens, inp.block_table, inp.num_q_heads, inp.num_kv_heads, inp.head_dim,
                        inp.max_pages, inp.num_pool_pages, inp.kv_dtype)
    assert p.plan.total_splits > inp.batch  # the scratch's split partials are exercised
    ref_out, ref_lse = ops.decode(p, q, kp, vp, bt, sl, inp.scale, ks, vs)
    assert B.pa_check_status(p.workspace) == B.PA_OK
    for _ in range(calls):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = B.pa_decode_noalloc(p.shapes, p.plan, q, kp, vp, ks, vs, bt, sl, p.meta_dev, inp.scale, out, lse)
        assert st == B.PA_OK
        _close(out, lse, ref_out, ref_lse, max_tol, mean_tol)


def test_noalloc_matches_pa_decode_on_two_calls_in_a_row():
    inp = W.make_decode(16, 32, 8, 128, W.uniform_lengths(21, 16, 1, 4096), seed=21)
    _check_against_pa_decode(inp, calls=2, max_tol=1e-2, mean_tol=1e-3)


def test_noalloc_after_a_different_call_e4m3():
    lens = W.lognormal_lengths(22, 12, math.log(1500.0), 1.0, 64, 6000)
    inp = W.make_decode(12, 64, 8, 128, lens, seed=22, kv_dtype="e4m3")
    _check_against_pa_decode(inp, calls=2, max_tol=5e-2, mean_tol=5e-3)


def test_noalloc_matches_the_oracle_and_reports_a_clean_status():
    """Two calls in a row against the fp64 oracle (same tolerances as every
    decode test: max |out| error 1e-2, mean 1e-3, lse 1e-3), each reading the
    device status word back through status_host."""
    inp = W.make_decode(10, 16, 4, 128, W.uniform_lengths(23, 10, 1, 3000), seed=23)
    q, kp, vp, ks, vs, bt, sl = _device_inputs(inp)
    p = ops.plan_decode(inp.seq_lens, inp.block_table, inp.num_q_heads, inp.num_kv_heads, inp.head_dim,
                        inp.max_pages, inp.num_pool_pages, inp.kv_dtype)
    assert p.plan.total_splits > inp.batch
    ref_out, ref_lse = oracle.decode(inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.seq_lens, inp.scale)
    for _ in range(2):
        out = torch.full((inp.batch, inp.num_q_heads, inp.head_dim), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((inp.batch, inp.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
        st = B.pa_decode_noalloc(p.shapes, p.plan, q, kp, vp, ks, vs, bt, sl, p.meta_dev, inp.scale, out, lse)
        assert st == B.PA_OK
        err = np.abs(out.float().cpu().numpy() - ref_out)
        assert err.max() <= 1e-2 and err.mean() <= 1e-3
        assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 1e-3


def test_noalloc_reports_a_device_fault_through_status_host():
    """An out-of-range page id in a live block-table slot is recorded by the
    kernel (the load is skipped, nothing faults) and comes back through
    status_host; the next clean call clears the word and reports PA_OK."""
    inp = W.make_decode(4, 8, 4, 128, [100, 700, 1500, 2100], seed=24)
    q, kp, vp, ks, vs, bt, sl = _device_inputs(inp)
    p = ops.plan_decode(inp.seq_lens, inp.block_table, inp.num_q_heads, inp.num_kv_heads, inp.head_dim,
                        inp.max_pages, inp.num_pool_pages, inp.kv_dtype)
    bad = inp.block_table.copy()
    bad[2, 5] = inp.num_pool_pages + 7  # 1500 keys: 24 pages, slot 5 is live
    bad_d = torch.from_numpy(bad).to("cuda")
    out = torch.empty((inp.batch, inp.num_q_heads, inp.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((inp.batch, inp.num_q_heads), dtype=torch.float32, device="cuda")
    st = B.pa_decode_noalloc(p.shapes, p.plan, q, kp, vp, ks, vs, bad_d, sl, p.meta_dev, inp.scale, out, lse)
    assert st == B.PA_ERR_DEVICE_BOUNDS
    st = B.pa_decode_noalloc(p.shapes, p.plan, q, kp, vp, ks, vs, bt, sl, p.meta_dev, inp.scale, out, lse)
    assert st == B.PA_OK


def test_noalloc_checks_arguments_before_enqueuing_anything():
    """A call refused on the host (here a NULL query) returns its error
    before the status word is cleared or any kernel is enqueued; the next
    valid call runs normally."""
    inp = W.make_decode(2, 8, 4, 128, [100, 200], seed=25)
    q, kp, vp, ks, vs, bt, sl = _device_inputs(inp)
    p = ops.plan_decode(inp.seq_lens, inp.block_table, inp.num_q_heads, inp.num_kv_heads, inp.head_dim,
                        inp.max_pages, inp.num_pool_pages, inp.kv_dtype)
    out = torch.empty((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(B.PaError) as e:
        B.pa_decode_noalloc(p.shapes, p.plan, None, kp, vp, ks, vs, bt, sl, p.meta_dev, inp.scale, out, lse)
    assert e.value.status == B.PA_ERR_INVALID_ARG
    st = B.pa_decode_noalloc(p.shapes, p.plan, q, kp, vp, ks, vs, bt, sl, p.meta_dev, inp.scale, out, lse)
    assert st == B.PA_OK


def test_noalloc_rejects_plans_beyond_its_scratch():
    # 64 sequences of 64 pages each, forced to 64 splits: ~67 MB of partials
    lens = np.full(64, 4096, np.int32)
    bt = np.arange(64 * 64, dtype=np.int32).reshape(64, 64)
    p = ops.plan_decode(lens, bt, 32, 8, 128, 64, 64 * 64, "bf16", forced_splits=64)
    assert p.plan.workspace_bytes > (16 << 20)
    dev = "cuda"
    # the call is refused on the host before any of these buffers is touched
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((1, 8, 64, 128), dtype=torch.bfloat16, device=dev)
    out = torch.empty((64, 32, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((64, 32), dtype=torch.float32, device=dev)
    btd, sl = torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev)
    with pytest.raises(B.PaError) as e:
        B.pa_decode_noalloc(p.shapes, p.plan, q, kv, kv, None, None, btd, sl, p.meta_dev, 0.088, out, lse)
    assert e.value.status == B.PA_ERR_WORKSPACE and "fixed" in str(e.value)
