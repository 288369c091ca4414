"""Block tables from flat page-id lists on the GPU (pa_page_table_from_flat,
through the C ABI) against the oracle's restatement of MATE's
_build_page_table_from_flat_kv_indices: bit-exact, including the error cases
the kernel records in the status word and replay inside a CUDA graph."""
import os

import numpy as np
import pytest
import torch

from oracle import scheduler as S
from paged_kv_attention_fwd_gb300 import binding as B
from paged_kv_attention_fwd_gb300.build import build

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


def run(flat, lens, columns, ws=None):
    dev = "cuda"
    idx = torch.tensor(np.asarray(flat, np.int32), device=dev)
    kl = torch.tensor(np.asarray(lens, np.int32), device=dev)
    bt = torch.full((len(lens), columns), -7, dtype=torch.int32, device=dev)
    ws = torch.zeros(B.PA_STATUS_BYTES, dtype=torch.uint8, device=dev) if ws is None else ws
    B.pa_page_table_from_flat(idx, len(flat), kl, len(lens), columns, bt, ws)
    return bt.cpu().numpy(), B.pa_check_status(ws)


def test_hand_worked_fixture():
    lines = [l for l in open(os.path.join(GOLDEN, "page_table_from_flat.txt")) if l.strip()]
    lens = [int(x) for x in next(l for l in lines if l.startswith("# kv_lens:")).split(":")[1].split()]
    idx = [int(x) for x in next(l for l in lines if l.startswith("# kv_indices:")).split(":")[1].split()]
    rows = [[int(x) for x in l.split()] for l in lines if not l.startswith("#")]
    got, st = run(idx, lens, 3)
    assert st == B.PA_OK
    assert got.tolist() == rows


@pytest.mark.parametrize("batch,extra_cols", [(1, 0), (7, 3), (1000, 0), (8192, 1)])
def test_matches_oracle(batch, extra_cols):
    rng = np.random.default_rng(batch)
    lens = rng.integers(0, 3000, size=batch).astype(np.int32)
    lens[::5] = 0
    lens[1::7] = 64 * rng.integers(1, 10, size=len(lens[1::7]))
    counts = (lens.astype(np.int64) + 63) // 64
    flat = rng.permutation(int(counts.sum()) + 17)[: int(counts.sum())].astype(np.int32)
    cols = int(counts.max(initial=1)) + extra_cols
    got, st = run(flat, lens, cols)
    assert st == B.PA_OK
    assert np.array_equal(got, np.array(S.page_table_from_flat(flat, lens, columns=cols), np.int32))


@pytest.mark.parametrize("case", ["short_list", "long_list", "negative_len", "row_overflow"])
def test_device_checks(case):
    """Inputs the definition rejects: the kernel records PA_ERR_DEVICE_BOUNDS,
    reads no id past the list, and still writes every entry of the table."""
    lens = [70, 0, 200, 5]  # 2 + 0 + 4 + 1 = 7 pages
    flat = list(range(100, 107))
    cols = 4
    if case == "short_list":
        flat = flat[:5]
    elif case == "long_list":
        flat = flat + [999]
    elif case == "negative_len":
        lens = [70, -3, 200, 5]
    elif case == "row_overflow":
        cols = 3
    got, st = run(flat, lens, cols)
    assert st == B.PA_ERR_DEVICE_BOUNDS
    assert np.all(got != -7)  # every entry written
    counts = [max(0, (n + 63) // 64) for n in lens]
    start = 0
    for b, c in enumerate(counts):
        for j in range(cols):
            src = start + j
            want = flat[src] if j < c and src < len(flat) else 0
            assert got[b, j] == want
        start += c


def test_replays_in_a_cuda_graph():
    """Capture once; new lengths and ids written in place before each replay
    give the tables of the new inputs.  The list length is a launch argument,
    fixed at capture, so the replays keep the captured page total."""
    dev = "cuda"
    batch, cols, total = 64, 40, 900
    rng = np.random.default_rng(9)

    def draw():
        counts = np.zeros(batch, np.int64)
        left = total
        while left:
            b = int(rng.integers(batch))
            if counts[b] < cols:
                counts[b] += 1
                left -= 1
        lens = np.where(counts > 0, (counts - 1) * 64 + rng.integers(1, 65, size=batch), 0).astype(np.int32)
        return lens, rng.permutation(batch * cols)[:total].astype(np.int32)

    lens, flat = draw()
    kl = torch.from_numpy(lens).to(dev)
    idx = torch.from_numpy(flat).to(dev)
    bt = torch.empty((batch, cols), dtype=torch.int32, device=dev)
    ws = torch.zeros(B.PA_STATUS_BYTES, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        B.pa_page_table_from_flat(idx, total, kl, batch, cols, bt, ws, stream=side)  # warm-up outside the capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            B.pa_page_table_from_flat(idx, total, kl, batch, cols, bt, ws, stream=side)
    for _ in range(3):
        lens, flat = draw()
        kl.copy_(torch.from_numpy(lens))
        idx.copy_(torch.from_numpy(flat))
        g.replay()
        torch.cuda.synchronize()
        assert B.pa_check_status(ws) == B.PA_OK
        assert np.array_equal(bt.cpu().numpy(), np.array(S.page_table_from_flat(flat, lens, columns=cols), np.int32))
