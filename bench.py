#!/usr/bin/env python
"""Benchmark: attention forward over a paged KV cache on GB300.

Default workload (the headline): batched GQA decode -- B=64, Hq=32, Hk=8,
D=128, bf16 KV in 64-row pages, seq_lens uniform in [1, 4096], seed 0.  The
metric is decode KV-read bandwidth: the K+V page bytes the step must read
(sum_b ceil(len_b/64) * 64 * Hk * D * 2 bytes * 2) per second.

One step = one pass of the decode hot path over the batch: pa_decode, whose
single kernel gathers the pages, attends and merges the split-KV partials
(the host scheduler's metadata is an input resident in HBM, as in serving
where one schedule serves every layer; the end-to-end number recomputes it
every step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle as the reference arm

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-attn decode KV-read GB/s (%HBM peak); prefill TFLOP/s (%TC peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = (f"flushed between steps outside the events: {L2_FLUSH_BYTES >> 20} MiB written (twice L2), then read "
           "back, so that no line of the previous step and no dirty line is left in L2")


class L2Flush:
    """Write a buffer twice the size of L2, then read it back.  The write
    evicts the previous step's lines; the read evicts the write's own dirty
    lines, whose write-back would otherwise compete with the next timed
    step for HBM bandwidth."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.buf.zero_()
        torch.sum(self.buf, dim=0, out=self.out)


NOMINAL_L2_BYTES = 129_000_000


def l2_note_for(input_bytes: int, l2: int = NOMINAL_L2_BYTES) -> str:
    """The config's statement of the L2 policy for a workload whose steps read
    `input_bytes`: inputs of at least three times L2 need no flush (a step's
    first reads evict whatever the previous step left); smaller ones are
    flushed."""
    if input_bytes >= 3 * l2:
        return f"no flush between steps: inputs larger than L2 ({input_bytes / 1e6:.0f} MB read per step, over 3x L2)"
    return L2_NOTE


def l2_policy(dev, input_bytes: int):
    """Returns (callable run between steps, the config note), decided with the
    device's own L2 size."""
    import torch
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or NOMINAL_L2_BYTES)
    note = l2_note_for(input_bytes, l2)
    if note != l2_note_for(input_bytes):
        raise RuntimeError(f"the L2 policy for {input_bytes} B differs between this device's L2 ({l2} B) and "
                           f"the nominal {NOMINAL_L2_BYTES} B the reference arm states")
    return (NoFlush() if note != L2_NOTE else L2Flush(dev)), note


class NoFlush:
    """The between-steps action for inputs larger than L2: nothing."""

    def __call__(self):
        pass


def time_steps(K, step, flush, stream):
    """Mean device time of one step (ms) over K steps, from CUDA events on the
    launching stream.  Without a flush the K steps run back to back between
    one pair of events, so each launch may start its shared-memory prologue
    while the previous step's kernel drains, as in a serving loop (every
    kernel still waits for the one before it before touching memory).  With a
    flush each step has its own pair of events and the flush runs outside
    them.  The caller synchronises before and after."""
    import torch
    if isinstance(flush, NoFlush):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            step()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / K
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    ev[-1][1].synchronize()
    return sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(K)) / K


PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "paged_kv_attention_fwd_gb300", "csrc")


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile_name, files):
    """DRAM bytes per launch recorded by an ncu capture of this kernel, if the
    kernel source is unchanged since the capture (else None)."""
    path = os.path.join(PROFILES, profile_name)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith(("source_sha256", "dram_bytes_per_launch_full")):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256") != source_sha(files):
        return None
    try:
        return float(vals["dram_bytes_per_launch_full"])
    except (KeyError, ValueError):
        return None


def max_over_ranks(values, dist, device):
    """The max of each value over all ranks: the slowest rank sets the job's
    time.  Identity without a process group."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_value(units_per_rank, world, seconds):
    """Whole-job throughput under weak scaling: every rank processes the same
    units, all ranks' units over the (max-over-ranks) time."""
    return world * units_per_rank / seconds


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out_path = os.path.join("/tmp", f"pa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.out_path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.out_path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.out_path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                    power.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[3:7]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.out_path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "power_w_max": max(power),
                "samples": len(sm), "reasons": sorted(reasons)}


def gpu_index(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return local_rank


# ------------------------------------------------------------------ workloads

def decode_workload(name):
    from paged_kv_attention_fwd_gb300 import workloads as W
    if name == "decode_gqa":
        inp = W.gqa_decode(0)
        desc = ("batched GQA decode: B=64, Hq=32, Hk=8, D=128, bf16 KV, page 64, q_len 1, "
                "seq_lens uniform[1,4096], seed 0")
    elif name == "decode_gqa_fp16":
        inp = W.gqa_decode(0, kv_dtype="f16")
        desc = ("batched GQA decode, fp16 q / KV / out: B=64, Hq=32, Hk=8, D=128, page 64, q_len 1, "
                "seq_lens uniform[1,4096], seed 0")
    elif name == "decode_gqa_graph":
        inp = W.gqa_decode(0)
        desc = ("batched GQA decode (B=64, Hq=32, Hk=8, D=128, bf16, seq_lens uniform[1,4096], seed 0) as one "
                "CUDA-graph replay per step: metadata written on the device from device seq_lens, then decode")
    elif name == "decode_fp8":
        inp = W.fp8_long_decode(0)
        desc = ("long-context decode, e4m3 KV with per-KV-head fp32 scales: B=128, Hq=64, Hk=8, D=128, page 64, "
                "seq_lens lognormal(ln 2048, 1) clipped to [64,16384], seed 0")
    elif name == "decode_tiny":
        inp = W.tiny_decode(0)
        desc = "tiny paged decode: B=2, Hq=8, Hk=4, D=64, seq_lens {37,130}, 8-page pool, seed 0"
    else:
        raise ValueError(name)
    return inp, desc


def kv_bytes(inp):
    el = 1 if inp.kv_dtype == "e4m3" else 2
    pages = sum((int(s) + 63) // 64 for s in inp.seq_lens)
    full = pages * 64 * inp.num_kv_heads * inp.head_dim * el * 2
    exact = int(np.sum(inp.seq_lens)) * inp.num_kv_heads * inp.head_dim * el * 2
    return full, exact


def prefill_workload(name):
    from paged_kv_attention_fwd_gb300 import workloads as W
    if name == "prefill_paged":
        inp = W.chunked_prefill(0)
        desc = ("chunked causal prefill against the paged cache: B=8, H=32 (Hq=Hk), D=128, page 64, q_len 512 "
                "after a cached prefix U[0,8192], qo_offset = kv_len - q_len, seed 0")
    elif name == "prefill_paged_fp16":
        inp = W.chunked_prefill(0, dtype="f16")
        desc = ("chunked causal prefill against the paged cache, fp16 q / K / V / out: B=8, H=32, D=128, page 64, "
                "q_len 512 after a cached prefix U[0,8192], seed 0")
    elif name == "mixed":
        inp = W.mixed_batch(0)
        desc = ("mixed decode + prefill batch: the GQA decode workload's 64 single-token sequences (kv U[1,4096]) "
                "then the chunked-prefill workload's 8 x 512 new tokens after a prefix U[0,8192]; Hq=32, Hk=8, "
                "D=128, bf16, one paged pool, one pa_mixed call, seed 0")
    elif name == "prefill_mla":
        inp = W.mla_prefill(0)
        desc = ("MLA ragged causal prefill: 8 sequences L~U[512,4096], H=128, q 192 = 128 nope + 64 rope, "
                "k_rope [T,1,64] shared by all heads, v/out 128, scale 1/sqrt(192), seed 0")
    elif name == "prefill_mla_fp8":
        inp = W.mla_e4m3_prefill(0)
        desc = ("fp8 MLA ragged causal prefill: the MLA workload (8 sequences L~U[512,4096], H=128) with q_nope / "
                "k_nope in e4m3 + per-head fp32 scales (amax/448), q_rope / k_rope / v bf16, seed 0")
    elif name == "prefill_mla_rope_fp8":
        inp = W.mla_rope_e4m3_prefill(0)
        desc = ("MLA ragged causal prefill with an e4m3 rope key: the MLA workload (8 sequences L~U[512,4096], "
                "H=128) with k_rope [T,1,64] in e4m3 + one fp32 scale per token (amax/448), q / k_nope / v bf16, "
                "seed 0")
    else:
        raise ValueError(name)
    return inp, desc


def visible_pairs(inp, causal=True):
    """Per query row, the number of keys it attends (the algorithmic unit)."""
    out = []
    for b in range(inp.batch):
        ql = int(inp.cu_seqlens_q[b + 1] - inp.cu_seqlens_q[b])
        kl = int(inp.cu_seqlens_k[b + 1] - inp.cu_seqlens_k[b])
        off = int(inp.qo_offset[b]) if inp.qo_offset is not None else kl - ql
        i = np.arange(ql, dtype=np.int64)
        out.append(np.clip(np.minimum(kl, off + i + 1) if causal else np.full(ql, kl), 0, kl))
    return np.concatenate(out)


def prefill_flops(inp, causal=True):
    """2 flops per multiply-add in QK^T (depth Dqk) and PV (depth Dv), per visible (row, key, head)."""
    pairs = int(visible_pairs(inp, causal).sum())
    return pairs * inp.num_q_heads * (2 * inp.head_dim_qk + 2 * inp.head_dim_v)


def decode_input_bytes(inp):
    """Bytes a decode step reads from its inputs: K+V pages and the queries."""
    return kv_bytes(inp)[0] + inp.q.size * 2


def decode_config(inp, desc, world):
    """The workload as both arms state it (nothing here depends on the implementation)."""
    full, exact = kv_bytes(inp)
    return {"workload": desc, "batch": inp.batch, "num_q_heads": inp.num_q_heads, "num_kv_heads": inp.num_kv_heads,
            "head_dim": inp.head_dim, "page_size": 64, "kv_bytes_per_step": full, "kv_bytes_token_exact": exact,
            "l2": l2_note_for(decode_input_bytes(inp)), "parallelism": f"replicas x{world}"}


def prefill_config(inp, desc, world, extra=None):
    """The workload as both arms state it (nothing here depends on the implementation)."""
    nbytes = sum(np.asarray(a).nbytes for a in prefill_host_arrays(inp).values())
    cfg = {"workload": desc, "total_q": int(inp.cu_seqlens_q[-1]), "num_q_heads": inp.num_q_heads,
           "head_dim_qk": inp.head_dim_qk, "head_dim_v": inp.head_dim_v, "flops_per_step": prefill_flops(inp),
           "l2": l2_note_for(nbytes), "parallelism": f"replicas x{world}"}
    cfg.update(extra or {})
    return cfg


# ------------------------------------------------------------------ reference arm (the oracle)

def cpu_oracle_decode_sample(inp, budget_s=None, steps=None, warmup=0):
    """Time the fp64 oracle on one sequence per step (cycling the batch).
    With budget_s: run until the budget is spent.  Returns (GB/s, seconds,
    sequences done, bytes)."""
    import oracle
    order = list(range(inp.batch))

    def one(b):
        sub = slice(b, b + 1)
        oracle.decode(inp.q[sub], inp.k_pool, inp.v_pool, inp.block_table[sub], inp.seq_lens[sub], inp.scale,
                      inp.kv_dtype, inp.k_scale, inp.v_scale)
        el = 1 if inp.kv_dtype == "e4m3" else 2
        return ((int(inp.seq_lens[b]) + 63) // 64) * 64 * inp.num_kv_heads * inp.head_dim * el * 2

    for i in range(warmup):
        one(order[i % len(order)])
    done, nbytes = 0, 0
    t0 = time.perf_counter()
    while True:
        nbytes += one(order[done % len(order)])
        done += 1
        el = time.perf_counter() - t0
        if steps is not None and done >= steps:
            break
        if budget_s is not None and el >= budget_s and done >= 1:
            break
    return nbytes / el / 1e9, el, done, nbytes


def cpu_oracle_prefill_sample(inp, budget_s=None, steps=None, warmup=0, rows_per_step=64, seed=0):
    """Time the fp64 oracle on random query rows (token, head) of the workload.
    Returns (TFLOP/s, seconds, rows done, flops)."""
    import oracle
    rng = np.random.default_rng(seed)
    pairs = visible_pairs(inp)
    hq = inp.num_q_heads
    per_pair = 2 * inp.head_dim_qk + 2 * inp.head_dim_v
    total_rows = pairs.size * hq

    def one():
        rows = rng.integers(0, total_rows, size=rows_per_step).astype(np.int64)
        if is_rope_fp8(inp):
            oracle.prefill_mla_rope_e4m3(inp.q, inp.k_nope, inp.v, inp.k_rope, inp.k_rope_scales, inp.cu_seqlens_q,
                                         inp.cu_seqlens_k, inp.scale, True, qo_offset=inp.qo_offset, rows=rows)
        elif is_fp8_mla(inp):
            oracle.prefill_mla_e4m3(inp.q_nope, inp.q_rope, inp.q_scale, inp.k_nope, inp.k_scale, inp.v, inp.k_rope,
                                    inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True, qo_offset=inp.qo_offset,
                                    rows=rows)
        else:
            oracle.prefill(inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k, inp.scale, True,
                           block_table=inp.block_table, k_rope=inp.k_rope, qo_offset=inp.qo_offset, rows=rows)
        return int(pairs[rows // hq].sum()) * per_pair

    for _ in range(warmup):
        one()
    done, flops = 0, 0
    t0 = time.perf_counter()
    while True:
        flops += one()
        done += 1
        el = time.perf_counter() - t0
        if steps is not None and done >= steps:
            break
        if budget_s is not None and el >= budget_s:
            break
    return flops / el / 1e12, el, done * rows_per_step, flops


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    cores = oracle.num_threads()
    if args.workload == "append":
        inp, prefix, qlen, kn, vn, desc = append_workload()
        for _ in range(args.warmup):
            oracle.append_kv(kn[:512], vn[:512], W_cu(qlen[:1]), prefix[:1], inp.block_table[:1], inp.k, inp.v)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle.append_kv(kn[:512], vn[:512], W_cu(qlen[:1]), prefix[:1], inp.block_table[:1], inp.k, inp.v)
        el = time.perf_counter() - t0
        gbs = args.steps * 4 * 512 * kn.shape[1] * 128 * 2 / el / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "implementation": "CPU oracle append",
                "config": {"workload": desc, "bytes_per_step": 4 * int(qlen.sum()) * kn.shape[1] * 128 * 2,
                           "l2": L2_NOTE, "parallelism": f"replicas x{args.gpus}"},
                "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                 "sample": "one sequence's 512 new tokens per step"},
                "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    if args.workload.startswith("prefill") or args.workload == "mixed":
        inp, desc = prefill_workload(args.workload)
        tfs, el, rows, flops = cpu_oracle_prefill_sample(inp, steps=args.steps, warmup=args.warmup, rows_per_step=8)
        line = {
            "impl": "reference", "metric": METRIC, "value": round(tfs, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "implementation": "fp64 CPU oracle (oracle/oracle.c), OpenMP",
            "config": prefill_config(inp, desc, args.gpus,
                                     {"num_decode": int(inp.meta["num_decode"])} if args.workload == "mixed" else None),
            "cpu_baseline": {"value": round(tfs, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": f"{rows} random (token, head) query rows, 8 per step"},
            "e2e": {"value": round(tfs, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return
    inp, desc = decode_workload(args.workload)
    gbs, el, done, nbytes = cpu_oracle_decode_sample(inp, steps=args.steps, warmup=args.warmup)
    sample = f"{done} single-sequence decode steps cycling the batch ({nbytes / 1e9:.3f} GB of K+V pages)"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / done * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "implementation": "fp64 CPU oracle (oracle/oracle.c), OpenMP",
        "config": decode_config(inp, desc, args.gpus),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def run_decode(args, rank, world, local_rank, dist):
    import torch
    from paged_kv_attention_fwd_gb300 import binding as B
    from paged_kv_attention_fwd_gb300 import ops

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp, desc = decode_workload(args.workload)
    full_bytes, exact_bytes = kv_bytes(inp)
    fp8 = inp.kv_dtype == "e4m3"
    f16 = inp.kv_dtype == "f16"
    graph = args.workload == "decode_gqa_graph"
    q = ops.as_16(inp.q, dev, "f16" if f16 else "bf16")
    conv = ops.as_e4m3 if fp8 else (lambda a, d: ops.as_16(a, d, "f16" if f16 else "bf16"))
    kp, vp = conv(inp.k_pool, dev), conv(inp.v_pool, dev)
    bt = torch.from_numpy(inp.block_table).to(dev)
    sl = torch.from_numpy(inp.seq_lens).to(dev)
    ks = torch.from_numpy(inp.k_scale).to(dev) if fp8 else None
    vs = torch.from_numpy(inp.v_scale).to(dev) if fp8 else None
    p = ops.plan_decode(inp.seq_lens, inp.block_table, inp.num_q_heads, inp.num_kv_heads, inp.head_dim,
                        inp.max_pages, inp.num_pool_pages, inp.kv_dtype, device=dev)
    out = torch.empty((inp.batch, inp.num_q_heads, inp.head_dim), dtype=torch.float16 if f16 else torch.bfloat16,
                      device=dev)
    lse = torch.empty((inp.batch, inp.num_q_heads), dtype=torch.float32, device=dev)
    flush, l2_note = l2_policy(dev, decode_input_bytes(inp))
    cfg = decode_config(inp, desc, world)
    assert cfg["l2"] == l2_note
    stream = torch.cuda.current_stream(dev)
    sh, plan = p.shapes, p.plan

    # the C call with its arguments marshalled once, as a serving loop would hold it
    step_call = B.prepared("pa_decode", sh, plan, q, kp, vp, ks, vs, bt, sl, p.meta_dev, ctypes.c_float(inp.scale),
                           out, lse, p.workspace, ctypes.c_size_t(p.workspace.numel()), stream=stream)

    if graph:
        # capture-safe form: a plan sized from capacities only, metadata written on
        # the device from device seq_lens, both launches captured in one CUDA graph
        # and replayed per step (new lengths would be written into `sl` in place)
        splan = B.pa_get_static_plan(sh)
        gmeta = torch.zeros(splan.meta_ints, dtype=torch.int32, device=dev)
        gws = torch.zeros(splan.workspace_bytes, dtype=torch.uint8, device=dev)
        stream = torch.cuda.Stream(dev)
        stream.wait_stream(torch.cuda.current_stream(dev))

        def eager():
            B.pa_get_metadata_device(sh, splan, sl, gmeta, stream=stream)
            B.pa_decode(sh, splan, q, kp, vp, ks, vs, bt, sl, gmeta, inp.scale, out, lse, gws, stream=stream)

        with torch.cuda.stream(stream):
            eager()  # the first launches configure the kernels outside the capture
        stream.synchronize()
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=stream):
            eager()
        p.workspace = gws

        def step_call():
            with torch.cuda.stream(stream):
                cg.replay()

    K = args.steps
    # the warm-up runs inside the sampler's window, after its settling pause,
    # so the timed steps follow it on a GPU that has not gone idle
    with ClockSampler(gpu_index(local_rank)) as clk:
        for _ in range(args.warmup):
            flush()
            step_call()
        torch.cuda.synchronize(dev)
        st = B.pa_check_status(p.workspace, stream)
        if st != B.PA_OK:
            raise RuntimeError(f"device status {st}: {B.pa_last_error()}")
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        ms = time_steps(K, step_call, flush, stream)  # a step: one decode launch, split merge fused in
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    kern_ms = ms
    ms, kern_ms = max_over_ranks([ms, kern_ms], dist, dev)
    st = B.pa_check_status(p.workspace, stream)
    if st != B.PA_OK:
        raise RuntimeError(f"device status {st}: {B.pa_last_error()}")
    clocks = clk.summary()

    pk, pk_src = peaks()
    value = job_value(full_bytes, world, ms * 1e-3) / 1e9
    achieved = full_bytes / (kern_ms * 1e-3) / 1e9
    kernel_files = ["decode.cu", "pa_ptx.cuh", "pa_internal.h", "pa_launch.h"]
    kname = "decode_f8_kernel" if fp8 and inp.head_dim == 128 else "decode_kernel"
    # the fp16 and graph-replayed forms run the same kernel over the same bytes as decode_gqa
    prof_wl = "decode_gqa" if args.workload in ("decode_gqa_fp16", "decode_gqa_graph") else args.workload
    prof = kname + "_" + prof_wl + ".md"
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": profiled_traffic(prof, kernel_files),
                "kernel": kname, "peak_source": f"{pk_src} (copy bandwidth)",
                "algorithmic_bytes_per_launch": full_bytes, "kernel_ms": round(kern_ms, 5)}

    e2e = None
    if not args.no_e2e:
        if graph:
            e2e = graph_decode_e2e(inp, dev, stream, cg, {"q": q, "k": kp, "v": vp, "bt": bt, "sl": sl}, out, lse,
                                   full_bytes, world, dist, args)
        else:
            e2e = decode_e2e(inp, dev, stream, sh, full_bytes, world, dist, args)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        gbs, el, done, nbytes = cpu_oracle_decode_sample(inp, budget_s=args.cpu_seconds)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{done} sequences of this batch through the fp64 oracle "
                         f"({nbytes / 1e9:.3f} GB of K+V pages, {el:.1f} s)"}
    launches = K * (2 if graph else 1)  # graph: the device scheduler and the decode kernel
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3+bf16" if fp8 else ("f16" if f16 else "bf16"), "data": "synthetic",
        "config": cfg,
        "schedule": {"splits": plan.total_splits, "ctas": plan.grid},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
    }
    return line


def graph_decode_e2e(inp, dev, stream, cg, dbuf, out, lse, full_bytes, world, dist, args):
    """End to end for the graph-replayed decode: every step copies all inputs
    from pinned memory into the captured buffers, replays the graph (device
    metadata + decode) and reads out + lse back."""
    import torch

    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()

    h = {"q": pinned(inp.q.view(np.int16)), "k": pinned(inp.k_pool.view(np.int16)),
         "v": pinned(inp.v_pool.view(np.int16)), "bt": pinned(inp.block_table), "sl": pinned(inp.seq_lens)}
    out_h = torch.empty(out.shape, dtype=torch.int16).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

    def step():
        with torch.cuda.stream(stream):
            for k in h:
                dbuf[k].view(h[k].dtype).copy_(h[k], non_blocking=True)
            cg.replay()
            out_h.copy_(out.view(torch.int16), non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
        torch.cuda.synchronize(dev)

    for _ in range(3):
        step()
    E = max(3, min(args.steps, args.e2e_steps))
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(E):
        step()
    el = time.perf_counter() - t0
    el, = max_over_ranks([el], dist, dev)
    h2d = sum(v.numel() * v.element_size() for v in h.values())
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    return {"value": round(world * full_bytes * E / el / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": E, "ms_per_step": round(el / E * 1e3, 4),
            "includes": "pinned H2D of all inputs + graph replay (device metadata + decode) + D2H of out/lse + sync"}


def decode_e2e(inp, dev, stream, sh, full_bytes, world, dist, args):
    """End to end through the public calls with host buffers: every step
    computes the schedule on the host, copies all inputs from pinned memory,
    runs pa_decode and reads out + lse back."""
    import torch
    from paged_kv_attention_fwd_gb300 import binding as B

    fp8 = inp.kv_dtype == "e4m3"

    def pinned(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t.pin_memory()

    h = {"q": pinned(inp.q.view(np.int16)), "k": pinned(inp.k_pool if fp8 else inp.k_pool.view(np.int16)),
         "v": pinned(inp.v_pool if fp8 else inp.v_pool.view(np.int16)), "bt": pinned(inp.block_table),
         "sl": pinned(inp.seq_lens)}
    if fp8:
        h["ks"], h["vs"] = pinned(inp.k_scale), pinned(inp.v_scale)
    d = {k: torch.empty_like(v, device=dev) for k, v in h.items()}
    meta0, plan0 = B.pa_get_metadata(inp.seq_lens, None, sh)
    meta_pin = torch.empty(plan0.meta_ints, dtype=torch.int32).pin_memory()
    meta_dev = torch.empty(plan0.meta_ints, dtype=torch.int32, device=dev)
    ws = torch.zeros(plan0.workspace_bytes, dtype=torch.uint8, device=dev)
    out_h = torch.empty((inp.batch, inp.num_q_heads, inp.head_dim), dtype=torch.int16).pin_memory()
    lse_h = torch.empty((inp.batch, inp.num_q_heads), dtype=torch.float32).pin_memory()
    out_d = torch.empty_like(out_h, device=dev)
    lse_d = torch.empty_like(lse_h, device=dev)
    sl_host = inp.seq_lens

    def step():
        meta, plan = B.pa_get_metadata(sl_host, None, sh)
        meta_pin.numpy()[: meta.size] = meta
        for k in h:
            d[k].copy_(h[k], non_blocking=True)
        meta_dev[: meta.size].copy_(meta_pin[: meta.size], non_blocking=True)
        B.pa_decode(sh, plan, d["q"], d["k"], d["v"], d.get("ks"), d.get("vs"), d["bt"], d["sl"], meta_dev,
                    inp.scale, out_d, lse_d, ws, stream=stream)
        out_h.copy_(out_d, non_blocking=True)
        lse_h.copy_(lse_d, non_blocking=True)
        torch.cuda.synchronize(dev)

    for _ in range(3):
        step()
    E = max(3, min(args.steps, args.e2e_steps))
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(E):
        step()
    el = time.perf_counter() - t0
    el, = max_over_ranks([el], dist, dev)
    h2d = sum(v.numel() * v.element_size() for v in h.values()) + plan0.meta_ints * 4
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    return {"value": round(world * full_bytes * E / el / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": E, "ms_per_step": round(el / E * 1e3, 4),
            "includes": "host schedule + pinned H2D of all inputs + pa_decode + D2H of out/lse + sync"}


def is_rope_fp8(inp):
    return hasattr(inp, "k_rope_scales")


def prefill_ws_bytes(inp, sh):
    from paged_kv_attention_fwd_gb300 import binding as B
    if is_rope_fp8(inp):
        return B.pa_prefill_mla_rope_fp8_workspace_size(sh)
    return B.pa_prefill_workspace_size(sh)


def is_fp8_mla(inp):
    return hasattr(inp, "q_nope")


def prefill_host_arrays(inp):
    """Name -> host array (16-bit elements as int16 bit patterns) of every input the call reads."""
    h = {"cq": inp.cu_seqlens_q, "ck": inp.cu_seqlens_k}
    if is_rope_fp8(inp):
        h.update(q=inp.q.view(np.int16), kn=inp.k_nope.view(np.int16), v=inp.v.view(np.int16), kr=inp.k_rope,
                 krs=inp.k_rope_scales)
        return h
    if is_fp8_mla(inp):
        h.update(qn=inp.q_nope, qr=inp.q_rope.view(np.int16), qs=inp.q_scale, kn=inp.k_nope, ks=inp.k_scale,
                 v=inp.v.view(np.int16), kr=inp.k_rope.view(np.int16))
        return h
    h.update(q=inp.q.view(np.int16), k=inp.k.view(np.int16), v=inp.v.view(np.int16))
    if inp.k_rope is not None:
        h["kr"] = inp.k_rope.view(np.int16)
    if inp.paged:
        h["bt"] = inp.block_table
    return h


def prefill_shapes_for(inp, dev):
    from paged_kv_attention_fwd_gb300 import binding as B
    from paged_kv_attention_fwd_gb300 import ops
    sh = ops.prefill_shapes(inp.batch, inp.num_q_heads, inp.num_kv_heads, inp.head_dim_qk, inp.head_dim_v,
                            inp.rope_dim, inp.max_seqlen_q, int(inp.cu_seqlens_q[-1]), int(inp.cu_seqlens_k[-1]),
                            max_pages=inp.block_table.shape[1] if inp.paged else 0,
                            num_pool_pages=inp.k.shape[0] if inp.paged else 0, device=dev)
    if is_fp8_mla(inp):
        sh.dtype = B.PA_KV_FP8_E4M3
    elif getattr(inp, "dtype", "bf16") == "f16":
        sh.dtype = B.PA_KV_FP16
    return sh


def prefill_launch(inp, sh, d, out, lse, ws, stream):
    """One call of the library's prefill entry for this workload on device buffers `d`."""
    from paged_kv_attention_fwd_gb300 import binding as B
    if is_rope_fp8(inp):
        B.pa_prefill_mla_rope_fp8(sh, d["q"], d["kn"], d["v"], d["kr"], d["krs"], d["cq"], d["ck"], None, True,
                                  inp.scale, out, lse, ws, stream=stream)
    elif is_fp8_mla(inp):
        B.pa_prefill_mla_fp8(sh, d["qn"], d["qr"], d["qs"], d["kn"], d["ks"], d["v"], d["kr"], d["cq"], d["ck"], None,
                             True, inp.scale, out, lse, ws, stream=stream)
    else:
        B.pa_prefill(sh, d["q"], d["k"], d["v"], d.get("kr"), d["cq"], d["ck"], d.get("bt"), None, True, inp.scale,
                     out, lse, ws, stream=stream)


def prefill_prepared(inp, sh, d, out, lse, ws, stream):
    """prefill_launch as one C call with its arguments marshalled once."""
    from paged_kv_attention_fwd_gb300 import binding as B
    nb = ctypes.c_size_t(ws.numel())
    sc = ctypes.c_float(inp.scale)
    if is_rope_fp8(inp):
        return B.prepared("pa_prefill_mla_rope_fp8", sh, d["q"], d["kn"], d["v"], d["kr"], d["krs"], d["cq"], d["ck"],
                          None, 1, sc, out, lse, ws, nb, stream=stream)
    if is_fp8_mla(inp):
        return B.prepared("pa_prefill_mla_fp8", sh, d["qn"], d["qr"], d["qs"], d["kn"], d["ks"], d["v"], d["kr"],
                          d["cq"], d["ck"], None, 1, sc, out, lse, ws, nb, stream=stream)
    return B.prepared("pa_prefill", sh, d["q"], d["k"], d["v"], d.get("kr"), d["cq"], d["ck"], d.get("bt"), None, 1,
                      sc, out, lse, ws, nb, stream=stream)


def prefill_device(inp, dev):
    import torch
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in prefill_host_arrays(inp).items()}
    return d, prefill_shapes_for(inp, dev)


def run_prefill(args, rank, world, local_rank, dist):
    import torch
    from paged_kv_attention_fwd_gb300 import binding as B

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp, desc = prefill_workload(args.workload)
    flops = prefill_flops(inp)
    d, sh = prefill_device(inp, dev)
    tq = int(inp.cu_seqlens_q[-1])
    out = torch.empty((tq, inp.num_q_heads, inp.head_dim_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((tq, inp.num_q_heads), dtype=torch.float32, device=dev)
    ws = torch.zeros(prefill_ws_bytes(inp, sh), dtype=torch.uint8, device=dev)
    flush, l2_note = l2_policy(dev, sum(t.numel() * t.element_size() for t in d.values()))
    cfg = prefill_config(inp, desc, world)
    assert cfg["l2"] == l2_note
    stream = torch.cuda.current_stream(dev)

    step = prefill_prepared(inp, sh, d, out, lse, ws, stream)

    K = args.steps
    with ClockSampler(gpu_index(local_rank)) as clk:  # warm-up inside the window, as for the decode
        for _ in range(args.warmup):
            flush()
            step()
        torch.cuda.synchronize(dev)
        if B.pa_check_status(ws, stream) != B.PA_OK:
            raise RuntimeError(B.pa_last_error())
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        ms = time_steps(K, step, flush, stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    ms, = max_over_ranks([ms], dist, dev)
    if B.pa_check_status(ws, stream) != B.PA_OK:
        raise RuntimeError(B.pa_last_error())
    clocks = clk.summary()
    pk, pk_src = peaks()
    tfs = flops / (ms * 1e-3) / 1e12
    peak = pk["bf16_tflops"]
    peak_source = f"{pk_src} (cuBLAS bf16 GEMM, burst)"
    if is_fp8_mla(inp):
        # 256 of the 640 flops per visible pair (q_nope . k_nope) run on e4m3 at twice
        # the bf16 rate (the nominal dense ratio): the time-weighted peak is
        # 640 / (256 / 2 + 384) = 1.25 x the bf16 peak
        peak = round(1.25 * peak, 1)
        peak_source += " x 1.25: e4m3 share of the flops at the nominal 2x bf16 rate"
    # the fp16 chunked prefill runs the same kernel over the same bytes as prefill_paged
    prof = "prefill_kernel_" + ("prefill_paged" if args.workload == "prefill_paged_fp16" else args.workload) + ".md"
    roofline = {"bound": "tensor", "achieved": round(tfs, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(tfs / peak, 4),
                "traffic": profiled_traffic(prof, ["prefill.cu", "prefill_common.cuh", "pa_ptx.cuh", "pa_internal.h"]),
                "kernel": "prefill_kernel", "peak_source": peak_source,
                "algorithmic_flops_per_launch": flops, "kernel_ms": round(ms, 5)}
    e2e = None
    if not args.no_e2e:
        e2e = prefill_e2e(inp, dev, stream, sh, flops, world, dist, args)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        ctf, el, rows, cfl = cpu_oracle_prefill_sample(inp, budget_s=args.cpu_seconds)
        cpu = {"value": round(ctf, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{rows} random (token, head) query rows of this workload through the fp64 oracle "
                         f"({cfl / 1e9:.2f} GFLOP, {el:.1f} s)"}
    line = {
        "metric": METRIC, "value": round(world * tfs, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "data": "synthetic",
        "dtype": ("e4m3+bf16" if (is_fp8_mla(inp) or is_rope_fp8(inp))
                  else ("f16" if getattr(inp, "dtype", "bf16") == "f16" else "bf16")),
        "config": cfg,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        # per step: the ordering kernel (with the larger workspace), the rope key's
        # expansion (e4m3 rope key only) and the prefill kernel
        "gpu_launches": K * (1 + (B.pa_prefill_workspace_size(sh) > B.PA_STATUS_BYTES) + is_rope_fp8(inp)),
        "clocks": clocks,
    }
    return line


def prefill_e2e(inp, dev, stream, sh, flops, world, dist, args):
    """End to end through pa_prefill with host buffers: copy q, k, v (and rope
    key, offsets, block table) from pinned memory, run, read out + lse back."""
    import torch
    from paged_kv_attention_fwd_gb300 import binding as B

    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()

    h = {k: pinned(v) for k, v in prefill_host_arrays(inp).items()}
    d = {k: torch.empty_like(v, device=dev) for k, v in h.items()}
    tq = int(inp.cu_seqlens_q[-1])
    out_h = torch.empty((tq, inp.num_q_heads, inp.head_dim_v), dtype=torch.int16).pin_memory()
    lse_h = torch.empty((tq, inp.num_q_heads), dtype=torch.float32).pin_memory()
    out_d = torch.empty_like(out_h, device=dev)
    lse_d = torch.empty_like(lse_h, device=dev)
    ws = torch.zeros(prefill_ws_bytes(inp, sh), dtype=torch.uint8, device=dev)

    def step():
        for k in h:
            d[k].copy_(h[k], non_blocking=True)
        prefill_launch(inp, sh, d, out_d, lse_d, ws, stream)
        out_h.copy_(out_d, non_blocking=True)
        lse_h.copy_(lse_d, non_blocking=True)
        torch.cuda.synchronize(dev)

    for _ in range(3):
        step()
    E = max(3, min(args.steps, args.e2e_steps))
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(E):
        step()
    el = time.perf_counter() - t0
    el, = max_over_ranks([el], dist, dev)
    h2d = sum(v.numel() * v.element_size() for v in h.values())
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    return {"value": round(world * flops * E / el / 1e12, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": E, "ms_per_step": round(el / E * 1e3, 4),
            "includes": "pinned H2D of q, k, v, offsets (+ rope key / block table) + pa_prefill + D2H of out/lse + sync"}


def append_workload():
    """The chunked-prefill workload's new chunk (8 x 512 tokens, 32 KV heads,
    D=128, bf16) written into its pages after each cached prefix."""
    from paged_kv_attention_fwd_gb300 import workloads as W
    inp = W.chunked_prefill(0)
    prefix = inp.meta["prefix"]
    qlen = np.diff(inp.cu_seqlens_q).astype(np.int32)
    kn = W.bf16_normal_fast(0, 90, (int(qlen.sum()), inp.num_kv_heads, 128))
    vn = W.bf16_normal_fast(0, 91, (int(qlen.sum()), inp.num_kv_heads, 128))
    desc = ("paged KV append: the chunked-prefill workload's 8 x 512 new tokens, 32 KV heads, D=128, bf16, "
            "written after cached prefixes U[0,8192] through block_table, seed 0")
    return inp, prefix, qlen, kn, vn, desc


def run_append(args, rank, world, local_rank, dist):
    import torch
    from paged_kv_attention_fwd_gb300 import binding as B
    from paged_kv_attention_fwd_gb300 import ops

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp, prefix, qlen, kn, vn, desc = append_workload()
    T, hk = kn.shape[0], kn.shape[1]
    nbytes = 4 * T * hk * 128 * 2  # read K and V rows, write K and V rows
    kp, vp = ops.as_bf16(inp.k, dev), ops.as_bf16(inp.v, dev)
    knd, vnd = ops.as_bf16(kn, dev), ops.as_bf16(vn, dev)
    cu = torch.from_numpy(W_cu(qlen)).to(dev)
    sp = torch.from_numpy(prefix).to(dev)
    bt = torch.from_numpy(inp.block_table).to(dev)
    sh = B.pa_append_shapes(batch=len(qlen), num_kv_heads=hk, head_dim=128, page_size=64,
                            max_pages_per_seq=inp.block_table.shape[1], num_pool_pages=inp.k.shape[0], total_new=T,
                            kv_dtype=B.PA_KV_BF16)
    ws = torch.zeros(B.PA_STATUS_BYTES, dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        B.pa_append_kv(sh, knd, vnd, cu, sp, bt, kp, vp, None, None, ws, stream=stream)

    K = args.steps
    with ClockSampler(gpu_index(local_rank)) as clk:  # warm-up inside the window, as for the decode
        for _ in range(args.warmup):
            flush()
            step()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        ms = time_steps(K, step, flush, stream)
        torch.cuda.synchronize(dev)
    ms, = max_over_ranks([ms], dist, dev)
    if B.pa_check_status(ws, stream) != B.PA_OK:
        raise RuntimeError(B.pa_last_error())
    pk, pk_src = peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    # end to end: new rows from pinned host memory, append, status word back
    kh = torch.from_numpy(kn.view(np.int16)).pin_memory()
    vh = torch.from_numpy(vn.view(np.int16)).pin_memory()
    st_h = torch.empty(1, dtype=torch.int32).pin_memory()

    def e2e_step():
        knd.view(torch.int16).copy_(kh, non_blocking=True)
        vnd.view(torch.int16).copy_(vh, non_blocking=True)
        step()
        st_h.copy_(ws[:4].view(torch.int32), non_blocking=True)
        torch.cuda.synchronize(dev)

    e2e = None
    if not args.no_e2e:
        for _ in range(3):
            e2e_step()
        E = max(3, min(K, args.e2e_steps))
        t0 = time.perf_counter()
        for _ in range(E):
            e2e_step()
        el = time.perf_counter() - t0
        e2e = {"value": round(world * nbytes * E / el / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": 2 * T * hk * 128 * 2, "d2h_bytes_per_step": 4, "steps": E,
               "ms_per_step": round(el / E * 1e3, 4)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        cut = 2  # two sequences of the batch per oracle pass
        c_new = qlen[:cut]
        kn_s, vn_s = kn[: int(c_new.sum())], vn[: int(c_new.sum())]
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < min(args.cpu_seconds, 5.0) or n == 0:
            oracle.append_kv(kn_s, vn_s, W_cu(c_new), prefix[:cut], inp.block_table[:cut], inp.k, inp.v)
            n += 1
        cel = time.perf_counter() - t0
        cb = n * 4 * int(c_new.sum()) * hk * 128 * 2
        cpu = {"value": round(cb / cel / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} oracle appends of 2 sequences' new tokens (copies the pools each time; {cel:.1f} s)"}
    line = {
        "metric": METRIC, "value": round(world * gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": desc, "bytes_per_step": nbytes, "l2": L2_NOTE, "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / pk["hbm_gbs"], 4),
                     "traffic": profiled_traffic("append_kernel_append.md", ["append.cu", "pa_internal.h", "pa_launch.h"]),
                     "kernel": "append_kernel",
                     "peak_source": f"{pk_src} (copy bandwidth)", "algorithmic_bytes_per_launch": nbytes,
                     "kernel_ms": round(ms, 5)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K, "clocks": clk.summary(),
    }
    return line


def run_mixed(args, rank, world, local_rank, dist):
    """One pa_mixed call per step: the decode kernel on the batch's leading
    single-token sequences, the prefill kernel on the rest.  value = attention
    FLOPs over every visible (row, key, head) / step time (the unit the oracle
    arm can report too); the roofline is time-weighted: the decode part's K/V
    bytes at the HBM peak plus the prefill part's FLOPs at the bf16 peak."""
    import torch
    from paged_kv_attention_fwd_gb300 import binding as B
    from paged_kv_attention_fwd_gb300 import ops

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp, desc = prefill_workload("mixed")
    nd = int(inp.meta["num_decode"])
    hq, hk = inp.num_q_heads, inp.num_kv_heads
    kl = np.diff(inp.cu_seqlens_k).astype(np.int32)
    sh = B.pa_mixed_shapes(batch=inp.batch, num_q_heads=hq, num_kv_heads=hk, head_dim=128, page_size=64,
                           max_pages_per_seq=inp.block_table.shape[1], num_pool_pages=inp.k.shape[0],
                           kv_dtype=B.PA_KV_BF16, num_sms=ops.num_sms(dev), ctas_per_sm=0, forced_splits=0)
    meta, plan = B.pa_get_mixed_plan(inp.cu_seqlens_q, kl, inp.block_table, sh)
    if plan.num_decode != nd:
        raise RuntimeError(f"mixed plan split at {plan.num_decode}, expected {nd}")
    tq = int(inp.cu_seqlens_q[-1])
    d = {"q": ops.as_bf16(inp.q, dev), "k": ops.as_bf16(inp.k, dev), "v": ops.as_bf16(inp.v, dev),
         "bt": torch.from_numpy(inp.block_table).to(dev), "cq": torch.from_numpy(inp.cu_seqlens_q).to(dev),
         "ck": torch.from_numpy(inp.cu_seqlens_k).to(dev), "kl": torch.from_numpy(kl).to(dev),
         "meta": torch.from_numpy(meta).to(dev)}
    out = torch.empty((tq, hq, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((tq, hq), dtype=torch.float32, device=dev)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    dec_ws = (plan.decode.workspace_bytes + 255) // 256 * 256 if plan.num_decode else 0
    flush, l2_note = l2_policy(dev, sum(t.numel() * t.element_size() for t in d.values()))
    cfg = prefill_config(inp, desc, world, {"num_decode": nd})
    stream = torch.cuda.current_stream(dev)

    def step():
        B.pa_mixed(sh, plan, d["q"], d["k"], d["v"], d["bt"], d["cq"], d["ck"], d["kl"], d["meta"], inp.scale, out,
                   lse, ws, stream=stream)

    def check():
        for part in (ws, ws[dec_ws:]):
            if B.pa_check_status(part, stream) != B.PA_OK:
                raise RuntimeError(B.pa_last_error())

    K = args.steps
    with ClockSampler(gpu_index(local_rank)) as clk:  # warm-up inside the window, as for the decode
        for _ in range(args.warmup):
            flush()
            step()
        torch.cuda.synchronize(dev)
        check()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        ms = time_steps(K, step, flush, stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    ms, = max_over_ranks([ms], dist, dev)
    check()
    clocks = clk.summary()
    pk, pk_src = peaks()
    pairs = visible_pairs(inp)
    per_pair = hq * (2 * 128 + 2 * 128)
    flops = int(pairs.sum()) * per_pair
    pre_flops = int(pairs[nd:].sum()) * per_pair  # decode rows come first, one row per sequence
    dec_bytes = int(sum((int(n) + 63) // 64 for n in kl[:nd])) * 64 * hk * 128 * 2 * 2
    t_ideal = dec_bytes / (pk["hbm_gbs"] * 1e9) + pre_flops / (pk["bf16_tflops"] * 1e12)
    tfs = flops / (ms * 1e-3) / 1e12
    eff_peak = flops / t_ideal / 1e12
    roofline = {"bound": "tensor", "achieved": round(tfs, 2), "peak": round(eff_peak, 1), "unit": "TFLOP/s",
                "frac": round(t_ideal / (ms * 1e-3), 4), "traffic": None, "kernel": "decode_kernel + prefill_kernel",
                "peak_source": (f"{pk_src}: time-weighted -- the decode part's K/V bytes at the copy bandwidth plus "
                                f"the prefill part's FLOPs at the cuBLAS bf16 peak ({t_ideal * 1e6:.1f} us for the "
                                f"step); frac = that time / the measured step time"),
                "decode_kv_bytes": dec_bytes, "prefill_flops": pre_flops, "kernel_ms": round(ms, 5)}
    e2e = None
    if not args.no_e2e:
        h = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in (
            ("q", inp.q.view(np.int16)), ("k", inp.k.view(np.int16)), ("v", inp.v.view(np.int16)),
            ("bt", inp.block_table), ("cq", inp.cu_seqlens_q), ("ck", inp.cu_seqlens_k), ("kl", kl))}
        meta_pin = torch.empty(meta.size, dtype=torch.int32).pin_memory()
        out_h = torch.empty((tq, hq, 128), dtype=torch.int16).pin_memory()
        lse_h = torch.empty((tq, hq), dtype=torch.float32).pin_memory()

        def e2e_step():
            m, pl = B.pa_get_mixed_plan(inp.cu_seqlens_q, kl, None, sh)
            meta_pin.numpy()[: m.size] = m
            for k in h:
                d[k].view(h[k].dtype).copy_(h[k], non_blocking=True)
            d["meta"][: m.size].copy_(meta_pin[: m.size], non_blocking=True)
            B.pa_mixed(sh, pl, d["q"], d["k"], d["v"], d["bt"], d["cq"], d["ck"], d["kl"], d["meta"], inp.scale,
                       out, lse, ws, stream=stream)
            out_h.copy_(out.view(torch.int16), non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
            torch.cuda.synchronize(dev)

        for _ in range(3):
            e2e_step()
        E = max(3, min(K, args.e2e_steps))
        t0 = time.perf_counter()
        for _ in range(E):
            e2e_step()
        el = time.perf_counter() - t0
        el, = max_over_ranks([el], dist, dev)
        e2e = {"value": round(world * flops * E / el / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in h.values()) + meta.size * 4,
               "d2h_bytes_per_step": out_h.numel() * 2 + lse_h.numel() * 4, "steps": E,
               "ms_per_step": round(el / E * 1e3, 4),
               "includes": "host mixed plan + pinned H2D of all inputs + pa_mixed + D2H of out/lse + sync"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        ctf, el, rows, cfl = cpu_oracle_prefill_sample(inp, budget_s=args.cpu_seconds)
        cpu = {"value": round(ctf, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{rows} random (token, head) query rows of this batch through the fp64 oracle "
                         f"({cfl / 1e9:.2f} GFLOP, {el:.1f} s)"}
    line = {
        "metric": METRIC, "value": round(world * tfs, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": cfg,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        # per step: the decode kernel, the prefill ordering kernel and the prefill kernel
        "gpu_launches": K * 3, "clocks": clocks,
    }
    return line


SECONDARY = ("decode_fp8", "prefill_paged", "prefill_mla")


def run_workload(args, rank, world, local_rank, dist):
    """Run one workload; returns its JSON record (every rank)."""
    if args.workload.startswith("prefill"):
        return run_prefill(args, rank, world, local_rank, dist)
    if args.workload == "mixed":
        return run_mixed(args, rank, world, local_rank, dist)
    if args.workload == "append":
        return run_append(args, rank, world, local_rank, dist)
    return run_decode(args, rank, world, local_rank, dist)


def secondary_record(line):
    """A workload's record as it sits under the headline's "secondary" key."""
    keep = ("value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config", "schedule", "roofline",
            "cpu_baseline", "e2e", "gpu_launches", "clocks")
    return {k: line[k] for k in keep if k in line}


def release_device_memory():
    import gc

    import torch
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def W_cu(lengths):
    from paged_kv_attention_fwd_gb300 import workloads as W
    return W.cu_seqlens(lengths)


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_gqa",
                    choices=["decode_gqa", "decode_gqa_fp16", "decode_gqa_graph", "decode_fp8", "decode_tiny",
                             "prefill_paged", "prefill_paged_fp16", "prefill_mla", "prefill_mla_fp8",
                             "prefill_mla_rope_fp8", "mixed", "append"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="with the default workload, skip the e4m3 decode and the two prefill records")
    ap.add_argument("--secondary-cpu-seconds", type=float, default=4.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        run_reference(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        dist = tdist
    from paged_kv_attention_fwd_gb300.build import build
    if rank == 0 or world == 1:
        build()
    if dist is not None:
        dist.barrier()
    line = run_workload(args, rank, world, local_rank, dist)
    if args.workload == "decode_gqa" and not args.no_secondary:
        # the rest of the metric in the same process: the e4m3 long-context decode
        # and both prefill shapes, each timed under the headline's own protocol
        line["secondary"] = {}
        for wl in SECONDARY:
            sub = argparse.Namespace(**{**vars(args), "workload": wl, "cpu_seconds": args.secondary_cpu_seconds})
            line["secondary"][wl] = secondary_record(run_workload(sub, rank, world, local_rank, dist))
            release_device_memory()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
