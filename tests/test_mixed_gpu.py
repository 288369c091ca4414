"""Mixed decode + prefill batches on the GPU: pa_mixed (through the C ABI)
runs the leading single-token sequences through the decode kernel and the rest
through the prefill kernel; the whole ragged output must match the oracle's
prefill over the batch (a decode row is a one-row segment)."""
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


def mixed_gpu(inp, dtype="bf16"):
    """One pa_mixed call over a paged prefill input (its leading one-row
    sequences become the decode part); returns out, lse, the plan and both
    parts' status words."""
    dev = "cuda"
    hq, hk = inp.num_q_heads, inp.num_kv_heads
    kl = np.diff(inp.cu_seqlens_k).astype(np.int32)
    sh = B.pa_mixed_shapes(batch=inp.batch, num_q_heads=hq, num_kv_heads=hk, head_dim=128, page_size=64,
                           max_pages_per_seq=inp.block_table.shape[1], num_pool_pages=inp.k.shape[0],
                           kv_dtype=B.PA_KV_FP16 if dtype == "f16" else B.PA_KV_BF16, num_sms=ops.num_sms(),
                           ctas_per_sm=0, forced_splits=0)
    meta, plan = B.pa_get_mixed_plan(inp.cu_seqlens_q, kl, inp.block_table, sh)
    tq = int(inp.cu_seqlens_q[-1])
    out = torch.empty((tq, hq, 128), dtype=torch.float16 if dtype == "f16" else torch.bfloat16, device=dev)
    lse = torch.empty((tq, hq), dtype=torch.float32, device=dev)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    B.pa_mixed(sh, plan, ops.as_16(inp.q, dev, dtype), ops.as_16(inp.k, dev, dtype), ops.as_16(inp.v, dev, dtype),
               torch.from_numpy(inp.block_table).to(dev), torch.from_numpy(inp.cu_seqlens_q).to(dev),
               torch.from_numpy(inp.cu_seqlens_k).to(dev), torch.from_numpy(kl).to(dev),
               torch.from_numpy(meta).to(dev), inp.scale, out, lse, ws)
    # status words of both parts (decode workspace first, prefill after it)
    dec = (plan.decode.workspace_bytes + 255) // 256 * 256 if plan.num_decode else 0
    st = (B.pa_check_status(ws), B.pa_check_status(ws[dec:]))
    return out.float().cpu().numpy(), lse.cpu().numpy(), plan, st


def run_mixed(q_lens, kv_lens, hq=8, hk=2, seed=60, dtype="bf16"):
    inp = W.make_paged_prefill(q_lens, kv_lens, hq, hk, 128, seed=seed, extra_pages=2, dtype=dtype)
    out, lse, plan, st = mixed_gpu(inp, dtype)
    ro, rl = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                            block_table=inp.block_table, dtype=dtype)
    return out, lse, ro, rl, plan, st


@pytest.mark.parametrize("q_lens,kv_lens", [
    ([1, 1, 1, 40, 300, 1, 128], [700, 1, 3000, 40, 1300, 65, 2000]),   # decode head, then mixed
    ([1] * 9, [5, 64, 65, 900, 4000, 1, 2, 129, 3000]),                  # decode only
    ([17, 1, 1, 256], [17, 100, 200, 1000]),                              # prefill from the first row
])
def test_mixed_batch_matches_oracle(q_lens, kv_lens):
    out, lse, ro, rl, plan, st = run_mixed(q_lens, kv_lens)
    assert st == (B.PA_OK, B.PA_OK)
    lead = 0
    while lead < len(q_lens) and q_lens[lead] == 1:
        lead += 1
    assert plan.num_decode == lead
    err = np.abs(out - ro)
    assert np.all(np.isfinite(out)) and err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(lse - rl).max() <= 1e-3


def test_mixed_batch_fp16():
    q_lens, kv_lens = [1, 1, 33, 1, 200], [900, 70, 100, 64, 1500]
    out, lse, ro, rl, plan, st = run_mixed(q_lens, kv_lens, seed=61, dtype="f16")
    assert st == (B.PA_OK, B.PA_OK) and plan.num_decode == 2
    err = np.abs(out - ro)
    assert np.all(np.isfinite(out)) and err.max() <= 1e-2 and err.mean() <= 1e-3
    assert np.abs(lse - rl).max() <= 1e-3


def test_mixed_full_size_sampled():
    """The bench's mixed step at full size (64 decodes of kv U[1,4096], then
    8 x 512-token chunks after a prefix U[0,8192]; Hq=32, Hk=8, D=128): every
    decode row and sampled rows of every chunk against the oracle."""
    from tests.test_prefill_gpu import sample_rows
    inp = W.mixed_batch(0)
    out, lse, plan, st = mixed_gpu(inp)
    assert st == (B.PA_OK, B.PA_OK) and plan.num_decode == 64
    rows = sample_rows(inp, per_seq=24)
    ro, rl = oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                            block_table=inp.block_table, rows=rows)
    hq = inp.num_q_heads
    o, l = out.reshape(-1, 128)[rows], lse.reshape(-1)[rows]
    assert np.all(np.isfinite(out))
    err = np.abs(o - ro)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3, f"max abs err {err.max():.3g}"
    assert np.abs(l - rl).max() <= 1e-3
    assert len({int(r) // hq for r in rows if int(r) // hq < 64}) == 64  # every decode row sampled
