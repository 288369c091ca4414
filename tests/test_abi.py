"""The C-ABI library without a GPU: it loads, exports every declared symbol,
its scheduler reproduces the oracle's scheduler bit for bit, and its host-side
validation rejects bad arguments with the documented status codes."""
import ctypes

import numpy as np
import pytest

from oracle import scheduler as S
from paged_kv_attention_fwd_gb300 import binding as B
from paged_kv_attention_fwd_gb300.build import build

from .test_scheduler_oracle import load_schedule_fixture


@pytest.fixture(scope="module", autouse=True)
def built():
    build()


def test_exports_every_declared_symbol():
    names = B.declared_symbols()
    assert {"pa_get_metadata", "pa_decode", "pa_prefill", "pa_check_status", "pa_last_error"} <= set(names)
    lib = B.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert B.pa_version() == 100


def shapes(B_, hq=32, hk=8, d=128, max_pages=64, pool=10**6, sms=152, cps=1, forced=0, kv=B.PA_KV_BF16):
    return B.pa_decode_shapes(batch=B_, num_q_heads=hq, num_kv_heads=hk, head_dim=d, page_size=64,
                              max_pages_per_seq=max_pages, num_pool_pages=pool, kv_dtype=kv, num_sms=sms,
                              ctas_per_sm=cps, forced_splits=forced)


def test_metadata_matches_hand_worked_fixture():
    g = load_schedule_fixture()
    sh = shapes(4, hq=4, hk=g["num_kv_heads"][0], max_pages=8, sms=g["num_sms"][0], cps=g["ctas_per_sm"][0],
                forced=g["forced_splits"][0])
    meta, plan = B.pa_get_metadata(np.array(g["seq_lens"], np.int32), None, sh)
    assert meta.tolist() == g["meta"]
    assert plan.total_splits == 5 and plan.num_items == 10 and plan.grid == 2


@pytest.mark.parametrize("case", range(12))
def test_metadata_bit_exact_against_oracle_scheduler(case):
    rng = np.random.default_rng(100 + case)
    if case % 3 == 0:
        lens = rng.integers(1, 4097, size=64)
        hk, sms, cps, maxp = 8, 152, 1 + case % 2, 64
    elif case % 3 == 1:
        lens = np.clip(np.floor(np.exp(np.log(2048) + rng.standard_normal(128))), 64, 16384).astype(int)
        hk, sms, cps, maxp = 8, 148, 1, 256
    else:
        lens = rng.integers(0, 300, size=int(rng.integers(1, 20)))
        hk, sms, cps, maxp = int(rng.integers(1, 5)), int(rng.integers(1, 9)), int(rng.integers(1, 3)), 5
    forced = [0, 0, 2, 7][case % 4]
    sh = shapes(len(lens), hq=hk * 2, hk=hk, max_pages=maxp, sms=sms, cps=cps, forced=forced)
    meta, plan = B.pa_get_metadata(lens.astype(np.int32), None, sh)
    ref = S.schedule(lens.tolist(), hk, sms, cps, forced)
    assert meta.tolist() == ref
    u = S.unpack(ref)
    assert plan.total_splits == u["total_splits"] and plan.grid == u["grid"] and plan.meta_ints == len(ref)
    assert plan.workspace_bytes >= 256 + u["total_splits"] * hk * 2 * 128 * 4


def test_metadata_sizing_call_and_small_capacity():
    sh = shapes(3)
    lens = np.array([5, 600, 4000], np.int32)
    plan = B.pa_decode_plan()
    lib = B.lib()
    assert lib.pa_get_metadata(lens.ctypes.data, None, ctypes.byref(sh), None, 0, ctypes.byref(plan)) == 0
    small = np.zeros(plan.meta_ints - 1, np.int32)
    st = lib.pa_get_metadata(lens.ctypes.data, None, ctypes.byref(sh), small.ctypes.data, small.size,
                             ctypes.byref(plan))
    assert st == B.PA_ERR_WORKSPACE and "capacity" in B.pa_last_error()


@pytest.mark.parametrize("mutate,needle", [
    (lambda s: setattr(s, "page_size", 128), "page_size"),
    (lambda s: setattr(s, "num_kv_heads", 0), "num_kv_heads"),
    (lambda s: setattr(s, "num_sms", 0), "num_sms"),
    (lambda s: setattr(s, "forced_splits", -1), "forced_splits"),
])
def test_metadata_rejects_bad_shapes(mutate, needle):
    sh = shapes(2)
    mutate(sh)
    with pytest.raises(B.PaError) as e:
        B.pa_get_metadata(np.array([10, 20], np.int32), None, sh)
    assert e.value.status == B.PA_ERR_INVALID_ARG and needle in str(e.value)


def test_metadata_rejects_long_sequence_and_bad_page_ids():
    sh = shapes(2, max_pages=2, pool=5)
    with pytest.raises(B.PaError, match="exceeds max_pages_per_seq"):
        B.pa_get_metadata(np.array([10, 129], np.int32), None, sh)
    with pytest.raises(B.PaError, match="negative"):
        B.pa_get_metadata(np.array([-1, 3], np.int32), None, sh)
    bt = np.array([[0, 1], [4, 5]], np.int32)  # row 1 slot 1 = 5 is outside [0, 5)
    with pytest.raises(B.PaError, match=r"block_table\[1, 1\]"):
        B.pa_get_metadata(np.array([10, 100], np.int32), bt, sh)
    # stale slot past ceil(len/64) is never checked (never read)
    B.pa_get_metadata(np.array([10, 64], np.int32), bt, sh)


class _Fake:
    """A non-null, 256-byte-aligned stand-in pointer; validation never dereferences it."""

    def __init__(self, addr=1 << 20, n=1 << 30):
        self.addr, self.n = addr, n

    def data_ptr(self):
        return self.addr

    def numel(self):
        return self.n

    def element_size(self):
        return 1


def _decode_call(sh, plan, **over):
    f = _Fake()
    args = dict(q=f, k_pool=f, v_pool=f, k_scale=None, v_scale=None, block_table=f, seq_lens=f, meta_dev=f,
                scale=0.1, out=f, lse=None, workspace=f)
    args.update(over)
    B.pa_decode(sh, plan, args["q"], args["k_pool"], args["v_pool"], args["k_scale"], args["v_scale"],
                args["block_table"], args["seq_lens"], args["meta_dev"], args["scale"], args["out"], args["lse"],
                args["workspace"], stream=1)


@pytest.mark.parametrize("mutate,over,status,needle", [
    (lambda s: setattr(s, "num_q_heads", 30), {}, B.PA_ERR_INVALID_ARG, "multiple"),
    (lambda s: setattr(s, "head_dim", 96), {}, B.PA_ERR_UNSUPPORTED, "head_dim"),
    (lambda s: (setattr(s, "num_q_heads", 8 * 32)), {}, B.PA_ERR_UNSUPPORTED, "group"),
    (lambda s: setattr(s, "kv_dtype", B.PA_KV_FP8_E4M3), {}, B.PA_ERR_INVALID_ARG, "k_scale"),
    (lambda s: None, {"q": None}, B.PA_ERR_INVALID_ARG, "NULL"),
    (lambda s: None, {"out": _Fake(addr=(1 << 20) + 8)}, B.PA_ERR_INVALID_ARG, "aligned"),
    (lambda s: None, {"scale": float("nan")}, B.PA_ERR_INVALID_ARG, "finite"),
    (lambda s: None, {"workspace": _Fake(n=100)}, B.PA_ERR_WORKSPACE, "workspace"),
])
def test_decode_host_validation(mutate, over, status, needle):
    sh = shapes(2, hq=32, hk=8)
    _, plan = B.pa_get_metadata(np.array([100, 300], np.int32), None, sh)
    mutate(sh)
    with pytest.raises(B.PaError) as e:
        _decode_call(sh, plan, **over)
    assert e.value.status == status and needle in str(e.value)


def test_wait_limit_validation():
    with pytest.raises(B.PaError):
        B.pa_set_wait_limit_ns(0)
    B.pa_set_wait_limit_ns(2_000_000_000)


def mixed_shapes(B_, hq=8, hk=2, max_pages=40, pool=10**5):
    return B.pa_mixed_shapes(batch=B_, num_q_heads=hq, num_kv_heads=hk, head_dim=128, page_size=64,
                             max_pages_per_seq=max_pages, num_pool_pages=pool, kv_dtype=B.PA_KV_BF16, num_sms=152,
                             ctas_per_sm=0, forced_splits=0)


def test_mixed_plan_splits_at_first_multi_token_segment():
    # MATE splits a mixed batch at the first sequence whose query length passes
    # its threshold; here the decode kernel takes the leading single-token rows
    cq = np.array([0, 1, 2, 3, 43, 44, 344], np.int32)  # q_len 1 1 1 40 1 300
    kl = np.array([10, 500, 1000, 100, 64, 400], np.int32)
    meta, plan = B.pa_get_mixed_plan(cq, kl, None, mixed_shapes(6))
    assert plan.num_decode == 3 and plan.total_q == 344 and plan.max_seqlen_q == 300
    assert meta.tolist() == S.schedule(kl[:3].tolist(), 2, 152, 1)  # decode part = the plain scheduler's plan
    # all-prefill and all-decode batches
    _, p2 = B.pa_get_mixed_plan(np.array([0, 5, 6], np.int32), np.array([5, 9], np.int32), None, mixed_shapes(2))
    assert p2.num_decode == 0 and p2.max_seqlen_q == 5
    _, p3 = B.pa_get_mixed_plan(np.array([0, 1, 2], np.int32), np.array([5, 9], np.int32), None, mixed_shapes(2))
    assert p3.num_decode == 2


def test_mixed_plan_rejects_more_queries_than_keys():
    with pytest.raises(B.PaError, match="query tokens"):
        B.pa_get_mixed_plan(np.array([0, 1, 30], np.int32), np.array([5, 9], np.int32), None, mixed_shapes(2))


def _mla_fp8_shapes(**over):
    d = dict(batch=2, num_q_heads=8, num_kv_heads=8, head_dim_qk=192, head_dim_v=128, rope_dim=64,
             max_seqlen_q=100, total_q=150, total_k=150, page_size=64, max_pages_per_seq=0, num_pool_pages=0,
             num_sms=152, dtype=B.PA_KV_FP8_E4M3)
    d.update(over)
    return B.pa_prefill_shapes(**d)


@pytest.mark.parametrize("over,args,status,needle", [
    ({"dtype": B.PA_KV_BF16}, {}, B.PA_ERR_INVALID_ARG, "PA_KV_FP8_E4M3"),
    ({"head_dim_qk": 128, "rope_dim": 0}, {}, B.PA_ERR_UNSUPPORTED, "192"),
    ({"num_q_heads": 6, "num_kv_heads": 4}, {}, B.PA_ERR_INVALID_ARG, "multiple"),
    ({}, {"q_scale": None}, B.PA_ERR_INVALID_ARG, "NULL"),
    ({}, {"k_rope": _Fake(addr=(1 << 20) + 4)}, B.PA_ERR_INVALID_ARG, "aligned"),
    ({}, {"scale": float("inf")}, B.PA_ERR_INVALID_ARG, "finite"),
    ({}, {"workspace": _Fake(n=16)}, B.PA_ERR_WORKSPACE, "workspace"),
])
def test_prefill_mla_fp8_host_validation(over, args, status, needle):
    f = _Fake()
    kw = dict(q_nope=f, q_rope=f, q_scale=f, k_nope=f, k_scale=f, v=f, k_rope=f, cu_seqlens_q=f, cu_seqlens_k=f,
              qo_offset=None, causal=True, scale=0.07, out=f, lse=None, workspace=f)
    kw.update(args)
    with pytest.raises(B.PaError) as e:
        B.pa_prefill_mla_fp8(_mla_fp8_shapes(**over), stream=1, **kw)
    assert e.value.status == status and needle in str(e.value)


def test_mixed_plan_rejects_e4m3_pools():
    # the prefill part has no e4m3-KV form: a mixed batch needs 16-bit pools
    sh = mixed_shapes(2)
    sh.kv_dtype = B.PA_KV_FP8_E4M3
    with pytest.raises(B.PaError) as e:
        B.pa_get_mixed_plan(np.array([0, 1, 30], np.int32), np.array([5, 90], np.int32), None, sh)
    assert e.value.status == B.PA_ERR_UNSUPPORTED and "pools" in str(e.value)


def _mla_rope_fp8_shapes(**over):
    d = dict(batch=2, num_q_heads=8, num_kv_heads=8, head_dim_qk=192, head_dim_v=128, rope_dim=64,
             max_seqlen_q=100, total_q=150, total_k=150, page_size=64, max_pages_per_seq=0, num_pool_pages=0,
             num_sms=152, dtype=B.PA_KV_BF16)
    d.update(over)
    return B.pa_prefill_shapes(**d)


def test_prefill_mla_rope_fp8_workspace_size():
    sh = _mla_rope_fp8_shapes()
    base = B.pa_prefill_workspace_size(sh)
    # pa_prefill's workspace rounded up to 256, then two rope levels of 150 * 128 bytes, each rounded up to 256
    assert B.pa_prefill_mla_rope_fp8_workspace_size(sh) == (base + 255) // 256 * 256 + 2 * ((150 * 128 + 255) // 256 * 256)


@pytest.mark.parametrize("over,args,status,needle", [
    ({"dtype": B.PA_KV_FP8_E4M3}, {}, B.PA_ERR_UNSUPPORTED, "PA_KV_BF16"),
    ({"head_dim_qk": 128, "rope_dim": 0}, {}, B.PA_ERR_UNSUPPORTED, "192"),
    ({"num_q_heads": 6, "num_kv_heads": 4}, {}, B.PA_ERR_INVALID_ARG, "multiple"),
    ({"total_k": 0}, {}, B.PA_ERR_INVALID_ARG, "total_k"),
    ({}, {"k_rope_scales": None}, B.PA_ERR_INVALID_ARG, "NULL"),
    ({}, {"k_rope": _Fake(addr=(1 << 20) + 8)}, B.PA_ERR_INVALID_ARG, "aligned"),
    ({}, {"k_rope_scales": _Fake(addr=(1 << 20) + 2)}, B.PA_ERR_INVALID_ARG, "4-byte"),
    ({}, {"scale": float("nan")}, B.PA_ERR_INVALID_ARG, "finite"),
    ({}, {"workspace": _Fake(n=4096)}, B.PA_ERR_WORKSPACE, "workspace"),
])
def test_prefill_mla_rope_fp8_host_validation(over, args, status, needle):
    f = _Fake(n=1 << 20)
    kw = dict(q=f, k_nope=f, v=f, k_rope=f, k_rope_scales=f, cu_seqlens_q=f, cu_seqlens_k=f, qo_offset=None,
              causal=True, scale=0.07, out=f, lse=None, workspace=f)
    kw.update(args)
    with pytest.raises(B.PaError) as e:
        B.pa_prefill_mla_rope_fp8(_mla_rope_fp8_shapes(**over), stream=1, **kw)
    assert e.value.status == status and needle in str(e.value)


@pytest.mark.parametrize("args,status,needle", [
    ({"batch": 0}, B.PA_ERR_UNSUPPORTED, "batch"),
    ({"batch": 8193}, B.PA_ERR_UNSUPPORTED, "batch"),
    ({"max_pages_per_seq": 0}, B.PA_ERR_INVALID_ARG, "max_pages_per_seq"),
    ({"num_indices": -1}, B.PA_ERR_INVALID_ARG, "num_indices"),
    ({"kv_lens": None}, B.PA_ERR_INVALID_ARG, "NULL"),
    ({"workspace": _Fake(n=16)}, B.PA_ERR_WORKSPACE, "workspace"),
])
def test_page_table_from_flat_host_validation(args, status, needle):
    f = _Fake()
    kw = dict(kv_indices=f, num_indices=10, kv_lens=f, batch=4, max_pages_per_seq=8, block_table=f, workspace=f)
    kw.update(args)
    with pytest.raises(B.PaError) as e:
        B.pa_page_table_from_flat(stream=1, **kw)
    assert e.value.status == status and needle in str(e.value)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without libpa.so every call raises: there is no CPU fallback."""
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "libpa.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        B.pa_version()
    sh = B.pa_decode_shapes(batch=1, num_q_heads=1, num_kv_heads=1, head_dim=64, page_size=64, max_pages_per_seq=1,
                            num_pool_pages=1, kv_dtype=B.PA_KV_BF16, num_sms=1, ctas_per_sm=0, forced_splits=0)
    with pytest.raises(RuntimeError, match="not built"):
        B.pa_get_metadata(np.array([1], np.int32), None, sh)


def test_product_path_never_imports_the_oracle():
    """The package's modules neither import nor load anything under oracle/."""
    import os
    import re
    pkg = os.path.dirname(B.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh")):
                src = open(os.path.join(root, f)).read()
                assert not re.search(r"^\s*(import oracle|from oracle)", src, re.M), f
                assert "liboracle" not in src and "oracle.c" not in src, f
