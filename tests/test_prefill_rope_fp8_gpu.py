"""MLA prefill with an e4m3 rope key on the GPU: pa_prefill_mla_rope_fp8 (through
the C ABI) against the fp64 oracle on the same seeded inputs.  Same tolerances
as the bf16 prefill: out max-abs 1e-2 and mean-abs 1e-3, lse abs 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_fwd_gb300 import binding as B
from paged_kv_attention_fwd_gb300 import ops
from paged_kv_attention_fwd_gb300 import workloads as W
from paged_kv_attention_fwd_gb300.build import build

from .parity import abs_values, assert_close_16
from .test_prefill_gpu import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


def run(inp, causal=True):
    out, lse, ws, _ = ops.prefill_mla_rope_fp8(inp, "cuda", causal=causal)
    st = B.pa_check_status(ws)
    return out.float().cpu().numpy(), lse.cpu().numpy(), st


def reference(inp, causal=True, rows=None):
    return oracle.prefill_mla_rope_e4m3(inp.q, inp.k_nope, inp.v, inp.k_rope, inp.k_rope_scales, inp.cu_seqlens_q,
                                        inp.cu_seqlens_k, inp.scale, causal, qo_offset=inp.qo_offset, rows=rows)


def test_mla_rope_fp8_ragged():
    inp = W.make_mla_rope_e4m3([50, 300, 513, 128, 1], 8, seed=21)
    out, lse, st = run(inp)
    assert st == B.PA_OK
    ro, rl = reference(inp)
    assert_close(out, lse, ro, rl)


@pytest.mark.parametrize("causal", [True, False])
def test_mla_rope_fp8_grouped_heads_and_explicit_offsets(causal):
    # query chunks after cached keys (kv_len > q_len), one with a negative offset
    inp = W.make_mla_rope_e4m3([40, 200, 130], 8, seed=22, num_kv_heads=2, kv_lens=[300, 200, 131],
                               causal=causal, qo_offset=[260, -5, 1])
    out, lse, st = run(inp, causal=causal)
    assert st == B.PA_OK
    ro, rl = reference(inp, causal=causal)
    assert_close(out, lse, ro, rl)


@pytest.mark.parametrize("kind", ["per_tensor", "some_zero", "spread", "large"])
def test_mla_rope_fp8_scale_shapes(kind):
    """One scale for every token (a per-tensor scale), zero scales, scales
    spread over 2^-3 .. 2^1 of the quantiser's, and scales 2^4 larger.  The
    last makes the softmax nearly one-hot, so an output is close to a single
    value row and its bf16 rounding alone can pass the absolute 1e-2 bar
    (half an ulp is 0.0156 on [4, 8)): that case is checked under the rule of
    tests/parity.py, the others under the stated bars."""
    inp = W.make_mla_rope_e4m3([130, 257], 4, seed=23)
    tk = inp.k_rope.shape[0]
    rng = np.random.default_rng(5)
    sc = {"per_tensor": np.full(tk, 0.0071, np.float32),
          "some_zero": np.where(np.arange(tk) % 7 == 0, 0.0, inp.k_rope_scales).astype(np.float32),
          "spread": (inp.k_rope_scales * np.exp2(rng.integers(-3, 2, size=tk))).astype(np.float32),
          "large": (inp.k_rope_scales * 16.0).astype(np.float32)}[kind]
    case = W.MlaRopeE4m3Inputs(**{**inp.__dict__, "k_rope_scales": sc})
    out, lse, st = run(case)
    assert st == B.PA_OK
    ro, rl = reference(case)
    if kind == "large":
        absv = W.MlaRopeE4m3Inputs(**{**case.__dict__, "v": abs_values(case.v)})
        abs_mean, _ = reference(absv)
        assert_close_16(out, lse, ro, rl, abs_mean)
    else:
        assert_close(out, lse, ro, rl)


def test_mla_rope_fp8_full_size_sampled():
    """The MLA workload's lengths and heads with an e4m3 rope key; every output
    checked finite, a sample of rows against the oracle."""
    inp = W.mla_rope_e4m3_prefill(0)
    out, lse, st = run(inp)
    assert st == B.PA_OK
    rng = np.random.default_rng(0)
    hq = inp.num_q_heads
    rows = []
    for b in range(inp.batch):
        a, e = int(inp.cu_seqlens_q[b]), int(inp.cu_seqlens_q[b + 1])
        pos = {0, 127, 128, 255, 256, e - a - 1} | set(rng.integers(0, e - a, size=20).tolist())
        for p in sorted(x for x in pos if x < e - a):
            for h in (0, hq // 2, hq - 1):
                rows.append((a + p) * hq + h)
    rows = np.array(rows, np.int64)
    ro, rl = reference(inp, rows=rows)
    assert_close(out.reshape(-1, 128)[rows], lse.reshape(-1)[rows], ro, rl)
    assert np.all(np.isfinite(out))


def test_mla_rope_fp8_repeats_bitwise():
    inp = W.make_mla_rope_e4m3([700, 65], 4, seed=24)
    o1, l1, _ = run(inp)
    o2, l2, _ = run(inp)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
