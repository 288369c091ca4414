"""The bench's multi-process logic on CPU: two gloo ranks (one process each,
as torchrun launches them) combine their step times by the max over ranks and
report the whole-job value; the reference arm does its work on rank 0 only.
Replicas only -- no collective is on the attention path, so this is the whole
N > 1 logic."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "..")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r took (10 + r) ms per step and (9 + r) ms of kernel time
    ms, kern = bench.max_over_ranks([10.0 + rank, 9.0 + rank], dist, "cpu")
    value = bench.job_value(1e9, world, ms * 1e-3)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms": ms, "kern": kern, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["ms"] == 11.0 and r["kern"] == 10.0       # the slowest rank's times, on every rank
        assert r["value"] == pytest.approx(2 * 1e9 / 11e-3)  # both ranks' units over that time


def test_single_process_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], None, "cpu") == [3.0, 4.0]
    assert bench.job_value(100.0, 1, 2.0) == 50.0


def test_reference_arm_runs_on_rank_0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "decode_tiny", "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_states_the_same_config_as_ours():
    """The reference arm's config is built by the same function as the GPU
    arm's (the workload only, nothing about the implementation)."""
    sys.path.insert(0, ROOT)
    import bench
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "decode_tiny", "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][0])
    inp, desc = bench.decode_workload("decode_tiny")
    assert line["config"] == bench.decode_config(inp, desc, 1)
    assert line["impl"] == "reference" and "implementation" not in line["config"]
