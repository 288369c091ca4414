"""bench.py's JSON line on the GPU: one short run of the default workload (with
the end-to-end and CPU-oracle legs) and one of a prefill workload, each line
checked for every key of the measurement contract."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3", *args],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def check_common(d, bound, unit):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and d["data"] == "synthetic"
    assert d["unit"] == unit and "workload" in d["config"]
    r = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r, key
    assert r["bound"] == bound and r["unit"] == unit and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert 0 < r["frac"] < 1.2
    assert d["gpu_launches"] >= d["steps"]
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and "reasons" in c


def check_legs(d, unit):
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == unit and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]


def test_default_line_with_e2e_cpu_baseline_and_secondary_records():
    d = run_bench("--cpu-seconds", "2", "--secondary-cpu-seconds", "1")
    check_common(d, "hbm", "GB/s")
    check_legs(d, "GB/s")
    assert d["gpu_launches"] == d["steps"]  # one decode launch a step
    # the rest of the metric, each record timed in the same process
    sec = d["secondary"]
    assert set(sec) == {"decode_fp8", "prefill_paged", "prefill_mla"}
    for name, r in sec.items():
        unit, bound = ("GB/s", "hbm") if name.startswith("decode") else ("TFLOP/s", "tensor")
        assert r["unit"] == unit and r["value"] > 0 and r["steps"] == 5 and r["ms_per_step"] > 0
        rf = r["roofline"]
        assert rf["bound"] == bound and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
        # achieved is recomputable from the record: algorithmic work / kernel time
        work = rf.get("algorithmic_flops_per_launch", rf.get("algorithmic_bytes_per_launch"))
        scale = 1e12 if unit == "TFLOP/s" else 1e9
        assert abs(work / (rf["kernel_ms"] * 1e-3) / scale - rf["achieved"]) <= 1e-3 * rf["achieved"] + 0.05
        check_legs(r, unit)
        assert "sm_mhz" in r["clocks"] and "workload" in r["config"]


def test_prefill_line():
    d = run_bench("--workload", "prefill_paged", "--no-e2e", "--no-cpu-baseline")
    check_common(d, "tensor", "TFLOP/s")
