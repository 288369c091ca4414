"""Pins for the oracle's split-KV scheduler: a hand-worked fixture and the
partition / balance properties the rule guarantees."""
import os

import numpy as np
import pytest

from oracle import scheduler as S
from paged_kv_attention_fwd_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load_schedule_fixture(name="schedule_small.txt"):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *rest = line.split()
            vals[key] = [int(x) for x in rest]
    return vals


def test_hand_worked_fixture():
    g = load_schedule_fixture()
    meta = S.schedule(g["seq_lens"], g["num_kv_heads"][0], g["num_sms"][0], g["ctas_per_sm"][0],
                      g["forced_splits"][0])
    assert meta == g["meta"]
    assert g["meta"][0] == 0x50414D31


def check_properties(seq_lens, hk, sms, cps, forced):
    meta = S.schedule(seq_lens, hk, sms, cps, forced)
    u = S.unpack(meta)
    assert u["length"] == len(meta)
    pages = [-(-max(s, 0) // 64) for s in seq_lens]
    n = u["n_splits"]
    assert u["split_indptr"][0] == 0 and u["split_indptr"][-1] == u["total_splits"] == sum(n)
    for b, p in enumerate(pages):
        assert 1 <= n[b] <= 64
        if forced > 0 and p > 1:
            assert n[b] == min(forced, p, 64)
        # splits tile [0, p) contiguously and in order, non-empty when p >= n
        ranges = [S.split_range(p, n[b], s) for s in range(n[b])]
        assert ranges[0][0] == 0 and ranges[-1][1] == p
        for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
            assert a1 == b0
        if p > 0:
            assert all(hi > lo for lo, hi in ranges)
    # every (b, s, kvh) appears exactly once
    want = {(b, s, k) for b in range(len(seq_lens)) for s in range(n[b]) for k in range(hk)}
    assert len(u["items"]) == len(want) and set(u["items"]) == want
    assert u["grid"] == min(len(want), sms * cps)
    # list scheduling bound: max load - min load <= max item cost
    cost = {}
    for b in range(len(seq_lens)):
        for s in range(n[b]):
            lo, hi = S.split_range(pages[b], n[b], s)
            for k in range(hk):
                cost[(b, s, k)] = hi - lo + 1
    cp = u["cta_indptr"]
    loads = [sum(cost[it] for it in u["items"][cp[c]:cp[c + 1]]) for c in range(u["grid"])]
    assert max(loads) - min(loads) <= max(cost.values())
    # items inside one CTA run longest first
    for c in range(u["grid"]):
        cs = [cost[it] for it in u["items"][cp[c]:cp[c + 1]]]
        assert cs == sorted(cs, reverse=True)
    return u


@pytest.mark.parametrize("forced", [0, 1, 2, 7])
def test_properties_uniform(forced):
    rng = np.random.default_rng(1)
    lens = rng.integers(1, 4097, size=64).tolist()
    check_properties(lens, 8, 152, 1, forced)


def test_properties_lognormal_and_edges():
    rng = np.random.default_rng(2)
    lens = np.clip(np.floor(np.exp(np.log(2048) + rng.standard_normal(128))), 64, 16384).astype(int)
    u = check_properties(lens.tolist(), 8, 152, 1, 0)
    assert u["total_splits"] > 128  # long sequences do get split
    check_properties([0, 0, 1, 64, 65, 128, 129], 3, 4, 2, 0)
    check_properties([16384] * 3, 1, 152, 1, 0)
    check_properties([5], 1, 1, 1, 0)


def test_deterministic():
    lens = list(range(0, 5000, 37))
    assert S.schedule(lens, 4, 152, 1) == S.schedule(lens, 4, 152, 1)


def test_snake_dealing_properties():
    rng = np.random.default_rng(7)
    lens = rng.integers(0, 8000, size=50).tolist()
    meta = S.schedule(lens, 4, 20, 1, dealing="snake")
    u = S.unpack(meta)
    lpt = S.unpack(S.schedule(lens, 4, 20, 1))
    assert u["n_splits"] == lpt["n_splits"] and sorted(u["items"]) == sorted(lpt["items"])
    cp = u["cta_indptr"]
    sizes = [cp[c + 1] - cp[c] for c in range(u["grid"])]
    assert max(sizes) - min(sizes) <= 1  # one item per CTA per round


def test_chunk_is_rounded_up_worked_by_hand():
    """One sequence of 1001 pages, one KV head, 10 CTAs: units / (2 items a
    CTA share x 10) = 1001 / 20 = 50.05, so chunk = 51 (rounded up, and above
    the floor of 4), and the sequence takes ceil(1001 / 51) = ceil(19.6) = 20
    splits of 50 or 51 pages."""
    u = S.unpack(S.schedule([1001 * 64], 1, 10, 1))
    assert u["chunk"] == 51
    assert u["n_splits"] == [20] and u["total_splits"] == 20
    widths = [hi - lo for lo, hi in (S.split_range(1001, 20, s) for s in range(20))]
    assert sorted(set(widths)) == [50, 51] and sum(widths) == 1001


def test_snake_dealing_worked_by_hand():
    """Six one-split sequences of 5, 4, 3, 2, 1 and 0 pages (one KV head, one
    split each): item costs 6, 5, 4, 3, 2, 1 (pages + 1), already longest
    first.  Three CTAs take them in the rounds 0, 1, 2 then 2, 1, 0, so CTA 0
    holds sequences 0 and 5, CTA 1 sequences 1 and 4, CTA 2 sequences 2 and 3:
    every CTA carries a cost of 7."""
    u = S.unpack(S.schedule([5 * 64, 4 * 64, 3 * 64, 2 * 64, 64, 0], 1, 3, 1, forced_splits=1, dealing="snake"))
    cp = u["cta_indptr"]
    per_cta = [[b for b, _, _ in u["items"][cp[c]:cp[c + 1]]] for c in range(3)]
    assert per_cta == [[0, 5], [1, 4], [2, 3]]


@pytest.mark.parametrize("hk,sms,cps,forced", [(8, 152, 1, 0), (1, 4, 2, 0), (3, 7, 1, 5)])
def test_static_capacity_bounds_every_length_mix(hk, sms, cps, forced):
    rng = np.random.default_rng(hk * 10 + sms)
    B = 40
    bound = S.static_split_capacity(B, hk, sms, cps, forced)
    for trial in range(200):
        kind = trial % 4
        if kind == 0:
            lens = rng.integers(0, 20000, size=B)
        elif kind == 1:
            lens = np.full(B, int(rng.integers(0, 300000)))
        elif kind == 2:
            lens = np.where(rng.random(B) < 0.1, 200000, 1)
        else:
            lens = rng.integers(0, 300, size=B)
        u = S.unpack(S.schedule(lens.tolist(), hk, sms, cps, forced))
        assert u["total_splits"] <= bound


# ---------------------------------------------------------------- block table from a flat page list

def test_page_table_from_flat_matches_the_hand_worked_fixture():
    lines = [l for l in open(os.path.join(GOLDEN, "page_table_from_flat.txt")) if l.strip()]
    lens = [int(x) for x in next(l for l in lines if l.startswith("# kv_lens:")).split(":")[1].split()]
    idx = [int(x) for x in next(l for l in lines if l.startswith("# kv_indices:")).split(":")[1].split()]
    rows = [[int(x) for x in l.split()] for l in lines if not l.startswith("#")]
    assert S.page_table_from_flat(idx, lens) == rows


def test_page_table_from_flat_round_trips_generated_block_tables():
    """Flattening the live entries of a generated block table row by row and
    rebuilding gives the table back (its unused entries are 0), for lengths with
    empty sequences and exact page multiples."""
    lens = np.array([0, 1, 63, 64, 65, 128, 1000, 4096, 7], np.int32)
    inp = W.make_decode(len(lens), 8, 8, 64, lens, seed=3)
    bt = inp.block_table
    flat = [int(bt[b, j]) for b in range(len(lens)) for j in range((int(lens[b]) + 63) // 64)]
    got = np.array(S.page_table_from_flat(flat, lens, columns=bt.shape[1]), np.int32)
    assert np.array_equal(got, bt)


def test_page_table_from_flat_rejects_mismatched_lists():
    with pytest.raises(ValueError):
        S.page_table_from_flat([1, 2], [65, 1])   # 3 pages implied
    with pytest.raises(ValueError):
        S.page_table_from_flat([], [-5])
    with pytest.raises(ValueError):
        S.page_table_from_flat([1, 2, 3], [130], columns=2)
