#!/usr/bin/env python
"""Benchmark of paged (block-sparse) KV-cache attention on one or more GB300s.

One step = one pass of the decode hot path over one batch of the
Llama-3-8B-shaped decode workload (batch 64, 32 q / 8 kv heads, head_dim 128,
page 16, bf16, kv_len ~ U[512, 4096], randomly permuted page pool): the host
plan (validation + equal-chunk split) with its copy to the device (a pipelined
plan: the copy overlaps the previous step's kernels), the split-KV decode kernel
and the log-sum-exp merge kernel, all through the C ABI.  Inputs are resident in
HBM; the KV read per step (~0.63 GB) is larger than L2, so no flush is needed
between steps.

The JSON line also carries the prefill (ragged causal, tensor cores), skewed
long-context decode (with and without the split), cascade, multi-level cascade,
append + RoPE, tree verification, mixed batch and column-vector prefill
measurements under "secondary".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own batch (weak scaling, no
collective on the data path); rank 0 prints the line.  --impl reference times
the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode KV GB/s & % of HBM peak; prefill TFLOP/s & % of tensor peak"
WORKLOAD = "llama3_8b_decode"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", default="own", choices=["own", "reference"])
    p.add_argument("--no-secondary", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--only", choices=["prefill", "prefill1", "cascade", "multilevel", "mixed", "append", "tree", "skewed",
                                      "tiny", "oracle"], default=None,
                   help="time one secondary measurement alone (for profiling) and print it")
    return p.parse_args()


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "paged_kv_cache_bsr_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(profile_name: str, src_hash: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith(("source_hash", "dram_bytes_per_launch",
                                                        "scale_to_bench_launch")):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_hash") != src_hash or "dram_bytes_per_launch" not in vals:
        return None
    return float(vals["dram_bytes_per_launch"]) * float(vals.get("scale_to_bench_launch", "1"))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not win and self.samples:  # a short window: take the samples nearest to it
            mid = 0.5 * (t0 + t1)
            win = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win)}


def combine_over_ranks(ms_per_step: float, nbytes: float):
    """Whole-job figures under torch.distributed: the slowest rank's step time and the
    bytes all ranks processed (each rank streams its own batch; no data moves between
    ranks).  Returns (max ms per step, total bytes)."""
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms_per_step], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    nb = torch.tensor([nbytes], dtype=torch.float64, device=dev)
    dist.all_reduce(nb, op=dist.ReduceOp.SUM)
    return float(t.item()), float(nb.item())


def rank_seed(rank: int) -> int:
    """Seed of the decode batch a rank streams (weak scaling: one batch per rank)."""
    return 1001 + rank


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    """The fp64 CPU oracle, as it stands, on the host cores: each step one bounded
    sample (a run of requests of the same workload, cycling through the batch)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from paged_kv_cache_bsr_gb300 import workloads as W
    oracle.build()
    b = W.llama3_decode(seed=1001)
    per_req = [n * 2 * b.num_kv_heads * b.head_dim * 2 for n in b.kv_lens]
    # Size one step so the whole run takes about two minutes at the oracle's speed.
    t = time.time()
    oracle.attention_of(b, rows=list(range(8)))
    rate = sum(per_req[:8]) / max(time.time() - t, 1e-6)  # bytes / s
    budget = 120.0 / max(args.steps + args.warmup, 1)
    n_req = max(1, min(b.batch, int(budget * rate / (sum(per_req) / b.batch))))
    cursor = [0]

    def step():
        rows = [(cursor[0] + i) % b.batch for i in range(n_req)]
        cursor[0] = (cursor[0] + n_req) % b.batch
        oracle.attention_of(b, rows=rows)
        return sum(per_req[r] for r in rows)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    nbytes = sum(step() for _ in range(args.steps))
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "batch": b.batch, "num_qo_heads": 32,
                                        "num_kv_heads": 8, "head_dim": 128, "page_size": 16,
                                        "kv_len": "U[512,4096]"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": f"{n_req} of {b.batch} requests per step, cycling"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- own arm
def cpu_baseline(b, seconds=10.0, single_core_seconds=3.0):
    """The oracle as it stands on the host cores over the whole batch, repeated ~10 s;
    then on one core over requests taken in turn, ~3 s."""
    import oracle
    oracle.build()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.attention_of(b)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    per_req = [n * 2 * b.num_kv_heads * b.head_dim * 2 for n in b.kv_lens]
    done, nbytes, t1 = 0, 0, time.perf_counter()
    while True:
        r = done % b.batch
        oracle.attention_of(b, rows=[r], threads=1)
        nbytes += per_req[r]
        done += 1
        if time.perf_counter() - t1 >= single_core_seconds:
            break
    dt1 = time.perf_counter() - t1
    return {"value": round(b.kv_bytes() * reps / dt / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"the full {WORKLOAD} batch (64 requests), {reps} passes, {dt:.1f} s",
            "single_core": {"value": round(nbytes / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                            "sample": f"{done} requests of the same batch in turn, {dt1:.1f} s"}}


def time_steps(fn, steps, warmup, stream, kernel_events=None, sync_each=False):
    """Device time of `steps` calls of fn on `stream` (CUDA events), after `warmup` calls."""
    import torch
    for _ in range(warmup):
        fn(None)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)] \
        if kernel_events else None
    start.record(stream)
    for k in range(steps):
        fn(pairs[k] if pairs else None)
    stop.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(stop)
    kern = None
    if pairs:
        kern = sum(a.elapsed_time(b) for a, b in pairs) / steps
    return total, kern


def host_plan_us(b, kind, reps=200):
    """Median host time of one plan step for batch b: pkv_plan_compute alone
    (validation and tables, no copy), on a host-only plan for this GPU's SM count."""
    import torch
    from paged_kv_cache_bsr_gb300 import api
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    params = api.make_params(b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.dtype, b.sm_scale,
                             b.logits_cap, b.causal)
    limits = api.Limits(max(b.batch, 1), max(b.total_q, 1), max(int(b.kv_indptr[-1]), 1))
    h = api.plan_create_host(kind, params, limits, sms)
    try:
        _, nbytes = api.plan_workspace_bytes(h)
        raw = torch.empty(nbytes + 64, dtype=torch.uint8)
        off = (-raw.data_ptr()) % 64
        ws = raw[off:off + nbytes]
        qo = b.qo_indptr if kind != api.PLAN_DECODE else None
        arrays = [api._host_i32(x) for x in (qo, b.kv_indptr, b.kv_indices, b.kv_last_page_len)]
        args = [api._ptr(x) for x in arrays] + [int(b.num_pages), api._ptr(ws), nbytes]
        lib = api.load()
        times = []
        for _ in range(reps):
            t0 = time.perf_counter()
            st = lib.pkv_plan_compute(h, b.batch, *args)
            times.append(time.perf_counter() - t0)
            if st != api.PKV_OK:
                raise api.PkvError(st, "pkv_plan_compute")
        return round(sorted(times)[len(times) // 2] * 1e6, 1)
    finally:
        api.plan_destroy(h)


def host_plan_or_error(b, kind):
    """host_plan_us, or the error it raised as text (recorded in place)."""
    try:
        return host_plan_us(b, kind)
    except Exception as e:
        return f"{type(e).__name__}: {e}"[:300]


def host_plan_entry(b):
    """The bench line's host plan figure for the decode batch."""
    from paged_kv_cache_bsr_gb300 import api
    return {"us": host_plan_or_error(b, api.PLAN_DECODE),
            "what": "pkv_plan_compute alone (validation + tables), median of 200 on the host; "
                    "the timed step's pipelined plan overlaps it with the GPU"}


def decode_measure(b, steps, warmup, peaks, profile_name=None, split_kv=True, kernel="decode_kernel"):
    """Step time and main-kernel time of plan + decode + merge on one workload
    (split_kv False: each page list whole on one worker, nothing to merge)."""
    import torch
    from paged_kv_cache_bsr_gb300 import runner, api
    db = runner.DeviceBatch.from_host(b)
    # A step loop re-plans every call: the pipelined plan copies each step's tables
    # while the previous step's kernels run.
    plan = runner.make_plan(b, api.PLAN_DECODE, pipelined=True, split_kv=split_kv)
    o = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.q.device)
    stream = torch.cuda.current_stream()

    def step(ev):
        if ev is not None:
            plan.set_timing_events(*ev)
        runner.plan_batch(plan, b)
        plan.run(db.q, db.kv_data, db.kv_indices, db.kv_indptr, db.kv_last_page_len, o, lse)

    # The step is timed plain; the main kernel's own time comes from a second, shorter
    # loop with events around it (events inside the step would add their own gaps).
    total_ms, _ = time_steps(step, steps, warmup, stream)
    _, kern_ms = time_steps(step, max(10, steps // 10), 3, stream, kernel_events=True)
    plan.set_timing_events(None, None)
    assert plan.device_error() == 0
    nbytes = b.kv_bytes()
    ms = total_ms / steps
    res = {"ms_per_step": ms, "kernel_ms": kern_ms, "bytes": nbytes, "value": nbytes / (ms * 1e-3) / 1e9,
           "info": plan.info()}
    traffic = recorded_traffic(profile_name, source_hash("decode.cu", "decode_kernel.cuh")) if profile_name else None
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    res["roofline"] = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                       "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                       "peak_source": peaks["source"], "kernel": kernel}
    del db, o, lse
    return res


def decode_e2e(b, steps):
    """The same metric through the C ABI with HOST buffers: every step copies q,
    the KV pool and the index arrays from pinned memory, plans, runs, and reads
    o and lse back."""
    import torch
    from paged_kv_cache_bsr_gb300 import runner, api
    dev = torch.device("cuda")
    pin = lambda t: t.contiguous().pin_memory()
    hq, hkv, hip, hix, hl = pin(b.q), pin(b.kv_data), pin(b.kv_indptr), pin(b.kv_indices), pin(b.kv_last_page_len)
    q = torch.empty_like(hq, device=dev)
    kv = torch.empty_like(hkv, device=dev)
    ip, ix, last = (torch.empty_like(t, device=dev) for t in (hip, hix, hl))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    ho = torch.empty_like(o, device="cpu").pin_memory()
    hlse = torch.empty_like(lse, device="cpu").pin_memory()
    plan = runner.make_plan(b, api.PLAN_DECODE)
    stream = torch.cuda.current_stream()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hkv, hip, hix, hl))
    d2h = ho.numel() * ho.element_size() + hlse.numel() * hlse.element_size()

    def step(_):
        for d, h in ((q, hq), (kv, hkv), (ip, hip), (ix, hix), (last, hl)):
            d.copy_(h, non_blocking=True)
        plan.plan(hip, hl, b.num_pages, kv_indices_h=hix)
        plan.run(q, kv, ix, ip, last, o, lse)
        ho.copy_(o, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    total_ms, _ = time_steps(step, steps, 3, stream)
    ms = total_ms / steps
    del q, kv, o
    return {"value": round(b.kv_bytes() / (ms * 1e-3) / 1e9, 3), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 4)}


def prefill_measure(peaks, steps=20, warmup=3, page_size=16):
    import torch
    from paged_kv_cache_bsr_gb300 import runner, api, workloads as W
    b = W.ragged_prefill(seed=1003, page_size=page_size)
    try:
        plan = runner.make_plan(b, api.PLAN_PREFILL, pipelined=True)
    except api.PkvError as e:
        return {"unavailable": str(e)}
    db = runner.DeviceBatch.from_host(b)
    o = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.q.device)

    def step(ev):
        if ev is not None:
            plan.set_timing_events(*ev)
        runner.plan_batch(plan, b)
        plan.run(db.q, db.kv_data, db.kv_indices, db.kv_indptr, db.kv_last_page_len, o, lse,
                 qo_indptr=db.qo_indptr)

    total_ms, _ = time_steps(step, steps, warmup, torch.cuda.current_stream())
    _, kern_ms = time_steps(step, steps, 2, torch.cuda.current_stream(), kernel_events=True)
    plan.set_timing_events(None, None)
    err = plan.device_error()
    if err:
        return {"workload": "ragged_causal_prefill", "page_size": page_size, "error": f"device error word {err}"}
    pairs = 0
    for qo, kv in zip(b.qo_lens, b.kv_lens):
        pre = kv - qo
        pairs += qo * pre + qo * (qo + 1) // 2
    flops = pairs * b.num_qo_heads * 4 * b.head_dim
    ms = total_ms / steps
    achieved = flops / (kern_ms * 1e-3) / 1e12
    # Pages of fewer than 8 rows: the timed span is the packing copy and the kernel
    # over it (the recorded ncu traffic is for 16-row pages only).
    packed = page_size < 8
    traffic = None if packed else recorded_traffic("prefill_kernel_ragged_causal_prefill.txt",
                                                   source_hash("prefill_kernel.cuh"))
    traffic = traffic if page_size == 16 else None
    return {"workload": "ragged_causal_prefill", "page_size": page_size,
            "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "kernel_ms": round(kern_ms, 4), "flops": flops,
            "host_plan_us": host_plan_or_error(b, api.PLAN_PREFILL),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": traffic,
                         "peak_source": peaks["source"],
                         "kernel": "pack_pages_kernel + prefill_kernel" if packed else "prefill_kernel"}}


def tree_measure(peaks, steps=20, warmup=3):
    """Speculative-decoding tree verification: 16 requests, prefix U[512, 4096], 64-node
    draft trees, custom-mask prefill; TFLOP/s over the query-key pairs the mask keeps."""
    import torch
    from paged_kv_cache_bsr_gb300 import runner, api, workloads as W
    tb = W.tree_verify(seed=1006)
    b = tb.batch
    plan = runner.make_plan(b, api.PLAN_PREFILL)
    db = runner.DeviceBatch.from_host(b)
    mask = tb.mask.cuda()
    o = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.q.device)
    runner.plan_batch(plan, b)

    def step(ev):
        if ev is not None:
            plan.set_timing_events(*ev)
        plan.run(db.q, db.kv_data, db.kv_indices, db.kv_indptr, db.kv_last_page_len, o, lse,
                 qo_indptr=db.qo_indptr, mask=mask)

    total_ms, _ = time_steps(step, steps, warmup, torch.cuda.current_stream())
    _, kern_ms = time_steps(step, steps, 2, torch.cuda.current_stream(), kernel_events=True)
    plan.set_timing_events(None, None)
    err = plan.device_error()
    if err:
        return {"workload": "tree_verify", "error": f"device error word {err}"}
    pairs = int(sum(int(m.sum()) for m in tb.matrices))
    flops = pairs * b.num_qo_heads * 4 * b.head_dim
    achieved = flops / (kern_ms * 1e-3) / 1e12
    kv_bytes = b.kv_bytes()
    return {"workload": "tree_verify", "requests": b.batch, "nodes": 64, "kernel_ms": round(kern_ms, 4),
            "ms_per_step": round(total_ms / steps, 4), "TFLOPs": round(achieved, 1),
            "tensor_frac": round(achieved / peaks["bf16_tflops"], 4),
            "kv_GBps": round(kv_bytes / (kern_ms * 1e-3) / 1e9, 1),
            "hbm_frac": round(kv_bytes / (kern_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "note": "64 query rows x 4 heads per kv head: one 256-row tile per (request, kv head); KV-read bound"}


PER_GRAPH = 10  # back-to-back calls per captured graph for the latency-bound secondaries


def graph_us(fn, s, steps, warmup, per_graph=1):
    """Capture ``per_graph`` back-to-back calls of fn on stream s in one CUDA graph;
    mean replay time in us divided by per_graph (per call: a graph replay's own launch
    cost, about 3 us on this GPU, is then spread over the calls, as it is over the many
    kernels of a model step)."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(per_graph):
            fn()
    with torch.cuda.stream(s):
        for _ in range(warmup):
            g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(steps):
            g.replay()
        b.record(s)
    b.synchronize()
    return round(a.elapsed_time(b) / steps / per_graph * 1e3, 2)


def tiny_measure(peaks, steps=50, warmup=5, per_graph=20):
    """The tiny fp16 decode (batch 4, 8 q / 2 kv heads, head_dim 64, page 16, kv_len
    U[1, 256], 64-page pool): launch-latency bound.  ``per_graph`` run calls (decode
    kernel + merge kernel each) are captured back to back in one CUDA graph and
    replayed, the plan made once outside; the figure is per call.  The decode kernel's
    own time comes from events around it (the plan's timing hook) in a plain loop."""
    import torch
    from paged_kv_cache_bsr_gb300 import runner, api, workloads as W
    b = W.tiny_decode(seed=1000)
    plan = runner.make_plan(b, api.PLAN_DECODE)
    db = runner.DeviceBatch.from_host(b)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        runner.plan_batch(plan, b, stream=s)
        o = torch.empty_like(db.q)
        lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device=db.q.device)
    s.synchronize()

    def run():
        plan.run(db.q, db.kv_data, db.kv_indices, db.kv_indptr, db.kv_last_page_len, o, lse, stream=s)

    def launches():
        for _ in range(per_graph):
            run()

    with torch.cuda.stream(s):
        launches()
    s.synchronize()
    us = graph_us(launches, s, steps, warmup) / per_graph

    def step(ev):
        if ev is not None:
            plan.set_timing_events(*ev)
        run()

    with torch.cuda.stream(s):
        _, kern_ms = time_steps(step, steps, warmup, s, kernel_events=True)
    plan.set_timing_events(None, None)
    err = plan.device_error()
    nbytes = b.kv_bytes()
    out = {"workload": "tiny_decode", "batch": b.batch, "kv_lens": list(b.kv_lens), "dtype": "fp16",
           "us_per_call": round(us, 2), "decode_kernel_us": round(kern_ms * 1e3, 2), "kv_bytes": nbytes,
           "kv_GBps": round(nbytes / (us * 1e-6) / 1e9, 2),
           "note": "latency bound (0.26 MB of K/V, fits in L2): GB/s is not a roofline figure here",
           "timing": f"CUDA-graph replay of {per_graph} back-to-back run calls; per-call time"}
    if err:
        out["error"] = f"device error word {err}"
    return out


def cascade_measure(peaks, steps=50, warmup=5):
    """Cascade (prefix prefill over one large row block + suffix decode + merge_state)
    vs non-cascade decode over prefix + suffix pages.  Plans are made once (the batch
    does not change); the run calls of each variant are captured in a CUDA graph and
    replayed, so the comparison is GPU time, not Python launch overhead."""
    import torch
    from paged_kv_cache_bsr_gb300 import runner, api, workloads as W
    cb = W.cascade_decode(seed=1004)
    try:
        pplan = runner.make_plan(cb.prefix, api.PLAN_PREFILL)
    except api.PkvError as e:
        return {"unavailable": str(e)}
    splan = runner.make_plan(cb.suffix, api.PLAN_DECODE)
    fplan = runner.make_plan(cb.full, api.PLAN_DECODE)
    kv = cb.full.kv_data.cuda()
    dp = runner.DeviceBatch.from_host(cb.prefix, kv_data=kv)
    ds = runner.DeviceBatch.from_host(cb.suffix, kv_data=kv)
    df = runner.DeviceBatch.from_host(cb.full, kv_data=kv)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        runner.plan_batch(pplan, cb.prefix, stream=s)
        runner.plan_batch(splan, cb.suffix, stream=s)
        runner.plan_batch(fplan, cb.full, stream=s)
        o_p = torch.empty_like(dp.q)
        l_p = torch.empty(dp.q.shape[:2], dtype=torch.float32, device=dp.q.device)
        o_s, l_s = torch.empty_like(o_p), torch.empty_like(l_p)
        o_f, l_f = torch.empty_like(o_p), torch.empty_like(l_p)

        def casc():
            pplan.run(dp.q, kv, dp.kv_indices, dp.kv_indptr, dp.kv_last_page_len, o_p, l_p,
                      qo_indptr=dp.qo_indptr, stream=s)
            splan.run(ds.q, kv, ds.kv_indices, ds.kv_indptr, ds.kv_last_page_len, o_s, l_s, stream=s)
            api.merge_state(o_p, l_p, o_s, l_s, o_p, l_p, stream=s)

        def full():
            fplan.run(df.q, kv, df.kv_indices, df.kv_indptr, df.kv_last_page_len, o_f, l_f, stream=s)

        casc()
        full()
    s.synchronize()
    # the same cascade as one mixed launch: prefix prefill beside the suffix decode
    m = W.cascade_as_mixed(cb.prefix, cb.suffix)
    dm = runner.DeviceBatch.from_host(m, kv_data=kv)
    mplan = runner.make_plan(m, api.PLAN_MIXED)
    with torch.cuda.stream(s):
        runner.plan_batch(mplan, m, stream=s)
        o_m = torch.empty_like(dm.q)
        l_m = torch.empty(dm.q.shape[:2], dtype=torch.float32, device=dm.q.device)
    B = cb.suffix.batch

    def casc_mixed():
        mplan.run(dm.q, kv, dm.kv_indices, dm.kv_indptr, dm.kv_last_page_len, o_m, l_m, qo_indptr=dm.qo_indptr,
                  stream=s)
        api.merge_state(o_m[B:], l_m[B:], o_m[:B], l_m[:B], o_m[B:], l_m[B:], stream=s)

    with torch.cuda.stream(s):
        casc_mixed()
    s.synchronize()
    out = {"workload": "cascade_softcap_decode"}
    for name, fn in (("cascade", casc), ("cascade_one_mixed_launch", casc_mixed), ("non_cascade", full)):
        out[name + "_us"] = graph_us(fn, s, steps, warmup, per_graph=PER_GRAPH)
        out[name + "_single_replay_us"] = graph_us(fn, s, steps, warmup)
    out["best_cascade_us"] = min(out["cascade_us"], out["cascade_one_mixed_launch_us"])
    out["speedup"] = round(out["non_cascade_us"] / out["best_cascade_us"], 3)
    out["non_cascade_kv_GBps"] = round(cb.full.kv_bytes() / (out["non_cascade_us"] * 1e-6) / 1e9, 1)
    # Unique K/V: the prefix once (one row block reads it for every request) plus every suffix.
    unique = cb.prefix.kv_bytes() + cb.suffix.kv_bytes()
    gbs = unique / (out["best_cascade_us"] * 1e-6) / 1e9
    out["roofline"] = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                       "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": None, "peak_source": peaks["source"],
                       "bytes": unique, "what": "unique K/V bytes (prefix once + suffixes) / best cascade time"}
    out["timing"] = (f"CUDA-graph replay of {PER_GRAPH} back-to-back run calls, per-call time (the *_single_replay_us "
                     "keys: one call per replay); plans made once outside the timed loop")
    return out


def multilevel_measure(steps=50, warmup=5):
    """Parallel generation over a three-level prefix tree (system prompt shared by 64
    requests, 8 prompts shared by 8 samples each, own generated tokens): the levels
    run in order on one stream, or concurrently on side streams, then merge_state;
    against non-cascade decode over every request's whole page list.  Each variant's
    run calls are replayed from a CUDA graph; plans are made once."""
    import torch
    from paged_kv_cache_bsr_gb300 import runner, api, workloads as W
    mb = W.parallel_generation(seed=1005)
    kv = mb.full.kv_data.cuda()
    levels = [runner.DeviceBatch.from_host(lv, kv_data=kv) for lv in mb.levels]
    df = runner.DeviceBatch.from_host(mb.full, kv_data=kv)
    s = torch.cuda.Stream()
    side = [torch.cuda.Stream() for _ in levels[1:]]
    try:
        plans = [runner.make_plan(lv, runner.level_kind(lv)) for lv in mb.levels]
    except api.PkvError as e:
        return {"unavailable": str(e)}
    fplan = runner.make_plan(mb.full, api.PLAN_DECODE)
    with torch.cuda.stream(s):
        for p, lv in zip(plans, mb.levels):
            runner.plan_batch(p, lv, stream=s)
        runner.plan_batch(fplan, mb.full, stream=s)
        o_f = torch.empty_like(df.q)
        l_f = torch.empty(df.q.shape[:2], dtype=torch.float32, device=df.q.device)

    def serial():
        runner.multi_level_cascade(levels, plans, stream=s)

    def concurrent():
        runner.multi_level_cascade(levels, plans, stream=s, side_streams=side)

    def full():
        fplan.run(df.q, kv, df.kv_indices, df.kv_indptr, df.kv_last_page_len, o_f, l_f, stream=s)

    # every level in one mixed launch (levels' rows listed again), then the merges
    m = W.levels_as_mixed(mb.levels)
    dm = runner.DeviceBatch.from_host(m, kv_data=kv)
    mplan = runner.make_plan(m, api.PLAN_MIXED)
    with torch.cuda.stream(s):
        runner.plan_batch(mplan, m, stream=s)
        o_m = torch.empty_like(dm.q)
        l_m = torch.empty(dm.q.shape[:2], dtype=torch.float32, device=dm.q.device)
    R, nl = mb.full.batch, len(mb.levels)

    def one_launch():
        mplan.run(dm.q, kv, dm.kv_indices, dm.kv_indptr, dm.kv_last_page_len, o_m, l_m, qo_indptr=dm.qo_indptr,
                  stream=s)
        # every level's states in one n-state merge, into the last level's rows
        api.merge_states(o_m, l_m, nl, o_m[(nl - 1) * R:], l_m[(nl - 1) * R:], stream=s)

    out = {"workload": "parallel_generation_3_level"}
    for name, fn in (("levels_serial", serial), ("levels_concurrent", concurrent), ("levels_one_mixed_launch",
                                                                                      one_launch),
                     ("non_cascade", full)):
        with torch.cuda.stream(s):
            fn()
        s.synchronize()
        out[name + "_us"] = graph_us(fn, s, steps, warmup, per_graph=PER_GRAPH)
        out[name + "_single_replay_us"] = graph_us(fn, s, steps, warmup)
    best = min(out["levels_serial_us"], out["levels_concurrent_us"], out["levels_one_mixed_launch_us"])
    out["speedup"] = round(out["non_cascade_us"] / best, 3)
    out["unique_kv_MB"] = round(sum(lv.kv_bytes() for lv in mb.levels) / 1e6, 1)
    out["non_cascade_kv_MB"] = round(mb.full.kv_bytes() / 1e6, 1)
    out["timing"] = (f"CUDA-graph replay of {PER_GRAPH} back-to-back run calls, per-call time (the *_single_replay_us "
                     "keys: one call per replay); plans made once outside the timed loop")
    return out


def append_bytes(b) -> int:
    """Algorithmic bytes of one append + RoPE launch: every new token's query read and
    written, its K and V read and written into the pool (index arrays not counted)."""
    e = b.kv_data.element_size()
    per_token = (2 * b.num_qo_heads + 4 * b.num_kv_heads) * b.head_dim * e
    return b.total_q * per_token


def append_measure(peaks, steps=50, warmup=5, per_graph=20):
    """Append stage with RoPE of keys and queries: the ragged prefill batch's new
    tokens (bandwidth: ~0.5 GB per launch, larger than L2) and one decode step of the
    Llama-3-8B-shaped batch (64 tokens, latency).  ``per_graph`` launches are captured
    in one CUDA graph and replayed, so host launch overhead is not timed; the figure
    is per launch."""
    import torch
    from paged_kv_cache_bsr_gb300 import runner, workloads as W
    out = {}
    for name, b in (("ragged_prefill_append", W.ragged_prefill(seed=1003)),
                    ("decode_step_append", W.llama3_decode(seed=1001))):
        k_new, v_new = W.new_kv_rows(b)
        db = runner.DeviceBatch.from_host(b)
        kn, vn = k_new.cuda(), v_new.cuda()
        q_out = torch.empty_like(db.q)
        s = torch.cuda.Stream()

        def launches():
            for _ in range(per_graph):
                runner.append_kv(db, kn, vn, 500000.0, q_out=q_out, stream=s)

        with torch.cuda.stream(s):
            launches()
        s.synchronize()
        us = graph_us(launches, s, steps, warmup) / per_graph
        nbytes = append_bytes(b)
        gbs = nbytes / (us * 1e-6) / 1e9
        out[name] = {"new_tokens": b.total_q, "us": round(us, 2), "bytes": nbytes, "GBps": round(gbs, 1),
                     "hbm_frac": round(gbs / peaks["hbm_gbs"], 4)}
        del db, kn, vn, q_out
    out["rope_theta"] = 500000.0
    out["timing"] = f"CUDA-graph replay of {per_graph} back-to-back launches; per-launch time"
    return out


def mixed_measure(steps=50, warmup=5):
    """A continuous-batching step of 60 decode requests and 4 prompt chunks: the mixed
    plan (one persistent launch, prefill CTAs beside decode CTAs on an SM split)
    against the two halves run back to back and against one prefill plan for every
    request (the 128-row tile for single-row requests too).  CUDA-graph replay of
    the run calls."""
    import torch
    from paged_kv_cache_bsr_gb300 import runner, api, workloads as W
    b = W.mixed_batch(seed=1007)
    dec = [r for r in range(b.batch) if b.qo_lens[r] == 1]
    pre = [r for r in range(b.batch) if b.qo_lens[r] > 1]
    bd, bp = W.sub_batch(b, dec), W.sub_batch(b, pre)
    kv = b.kv_data.cuda()
    db, dd, dp = (runner.DeviceBatch.from_host(x, kv_data=kv) for x in (b, bd, bp))
    pm = runner.make_plan(b, api.PLAN_MIXED)
    pd = runner.make_plan(bd, api.PLAN_DECODE)
    pp = runner.make_plan(bp, api.PLAN_PREFILL)
    pu = runner.make_plan(b, api.PLAN_PREFILL)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for plan, x in ((pm, b), (pd, bd), (pp, bp), (pu, b)):
            runner.plan_batch(plan, x, stream=s)
        outs = {k: (torch.empty_like(x.q), torch.empty(x.q.shape[:2], dtype=torch.float32, device="cuda"))
                for k, x in (("m", db), ("d", dd), ("p", dp), ("u", db))}

    def run(plan, x, k):
        o, lse = outs[k]
        plan.run(x.q, kv, x.kv_indices, x.kv_indptr, x.kv_last_page_len, o, lse, qo_indptr=x.qo_indptr, stream=s)

    variants = (("mixed", lambda: run(pm, db, "m")),
                ("sequential", lambda: (run(pd, dd, "d"), run(pp, dp, "p"))),
                ("decode_half_alone", lambda: run(pd, dd, "d")),
                ("prefill_half_alone", lambda: run(pp, dp, "p")),
                ("one_prefill_plan", lambda: run(pu, db, "u")))
    out = {"workload": "mixed_batch", "decode_requests": len(dec), "prefill_requests": len(pre),
           "prefill_rows": bp.total_q}
    for name, fn in variants:
        with torch.cuda.stream(s):
            fn()
        s.synchronize()
        out[name + "_us"] = graph_us(fn, s, steps, warmup)
    info = pm.info()
    out["prefill_ctas"], out["decode_ctas"] = info.prefill_ctas, info.decode_ctas
    out["speedup_vs_sequential"] = round(out["sequential_us"] / out["mixed_us"], 3)
    out["host_plan_us"] = host_plan_or_error(b, api.PLAN_MIXED)
    err = pm.device_error()
    if err:
        out["error"] = f"device error word {err}"
    out["timing"] = "CUDA-graph replay of the run calls; plans made once outside the timed loop"
    return out


def oracle_configs(seconds_per_config=8.0):
    """The fp64 CPU oracle as it stands on each of the five workloads, on the host
    cores: whole workloads (repeated until the time budget) where one pass is short,
    else the ragged prefill's query rows taken in order until the budget; each rate in
    the workload's own unit."""
    import oracle
    from paged_kv_cache_bsr_gb300 import workloads as W
    oracle.build()
    out = {"cores": oracle.num_threads()}

    def kv_rate(b):
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle.attention_of(b)
            reps += 1
            if time.perf_counter() - t0 >= seconds_per_config:
                break
        dt = time.perf_counter() - t0
        return {"GBps": round(b.kv_bytes() * reps / dt / 1e9, 4), "passes": reps, "s": round(dt, 2)}

    t = W.tiny_decode(seed=1000)
    t0 = time.perf_counter()
    oracle.attention_of(t)
    out["tiny_decode"] = {"us_per_call": round((time.perf_counter() - t0) * 1e6, 1)}
    for name, b in (("llama3_8b_decode", W.llama3_decode(seed=1001)), ("skewed_decode", W.skewed_decode(seed=1002))):
        out[name] = kv_rate(b)
    p = W.ragged_prefill(seed=1003)
    pairs_row = []
    for qo, kv in zip(p.qo_lens, p.kv_lens):
        pre = kv - qo
        pairs_row += [pre + i + 1 for i in range(qo)]
    done, t0 = 0, time.perf_counter()
    step = 256
    while time.perf_counter() - t0 < seconds_per_config and done < p.total_q:
        rows = list(range(done, min(done + step, p.total_q)))
        oracle.attention_of(p, rows=rows)
        done = rows[-1] + 1
    dt = time.perf_counter() - t0
    flops = sum(pairs_row[:done]) * p.num_qo_heads * 4 * p.head_dim
    out["ragged_causal_prefill"] = {"TFLOPs": round(flops / dt / 1e12, 5), "rows": done, "of": p.total_q,
                                    "s": round(dt, 2)}
    cb = W.cascade_decode(seed=1004)
    t0 = time.perf_counter()
    oracle.attention_of(cb.full)
    dt = time.perf_counter() - t0
    out["cascade_softcap_decode"] = {"us_per_call": round(dt * 1e6, 1),
                                     "what": "non-cascade attention over every request's full page list"}
    return out


def run_only(args):
    if args.only == "oracle":  # host cores only
        print(json.dumps({"only": "oracle", **oracle_configs()}), flush=True)
        return
    import torch
    from paged_kv_cache_bsr_gb300 import build, api, workloads as W
    torch.cuda.set_device(0)
    build.build()
    api.load()
    peaks = measured_peaks()
    if args.only == "prefill":
        res = prefill_measure(peaks, steps=args.steps, warmup=args.warmup)
    elif args.only == "prefill1":
        res = prefill_measure(peaks, steps=args.steps, warmup=args.warmup, page_size=1)
    elif args.only == "tiny":
        res = tiny_measure(peaks, steps=args.steps, warmup=args.warmup)
    elif args.only == "cascade":
        res = cascade_measure(peaks, steps=args.steps, warmup=args.warmup)
    elif args.only == "multilevel":
        res = multilevel_measure(steps=args.steps, warmup=args.warmup)
    elif args.only == "mixed":
        res = mixed_measure(steps=args.steps, warmup=args.warmup)
    elif args.only == "append":
        res = append_measure(peaks, steps=args.steps, warmup=args.warmup)
    elif args.only == "tree":
        res = {"tree": tree_measure(peaks, steps=args.steps, warmup=args.warmup),
               "page_size_1": prefill_measure(peaks, steps=args.steps, warmup=args.warmup, page_size=1)}
    else:
        sk = W.skewed_decode(seed=1002)
        r = decode_measure(sk, args.steps, args.warmup, peaks)
        r0 = decode_measure(sk, args.steps, args.warmup, peaks, split_kv=False)
        res = {"value": round(r["value"], 1), "unit": "GB/s", "roofline": r["roofline"],
               "split_off": {"value": round(r0["value"], 1), "ms_per_step": round(r0["ms_per_step"], 4),
                             "split_speedup": round(r0["ms_per_step"] / r["ms_per_step"], 2)}}
    print(json.dumps({"only": args.only, **res}), flush=True)


def run_own(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from paged_kv_cache_bsr_gb300 import build, api, workloads as W
    build.build()
    api.load()
    peaks = measured_peaks()
    b = W.llama3_decode(seed=rank_seed(rank))
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    res = decode_measure(b, args.steps, args.warmup, peaks, "decode_kernel_llama3_8b_decode.txt")
    t_wall1 = time.time()
    ms = res["ms_per_step"]
    if world > 1:
        ms, total_bytes = combine_over_ranks(ms, res["bytes"])
        dist.barrier()
    else:
        total_bytes = res["bytes"]
    clk = clocks.summary(t_wall0, t_wall1)
    if rank != 0:
        clocks.stop()
        if world > 1:
            dist.destroy_process_group()
        return
    value = total_bytes / (ms * 1e-3) / 1e9
    info = res["info"]
    secondary = {}
    e2e = None
    if world == 1:
        if args.e2e_steps > 0:
            e2e = decode_e2e(b, args.e2e_steps)
        if not args.no_secondary:
            sk = W.skewed_decode(seed=1002)
            r3 = decode_measure(sk, max(20, args.steps // 10), 5, peaks)
            secondary["skewed_decode"] = {"value": round(r3["value"], 1), "unit": "GB/s",
                                          "ms_per_step": round(r3["ms_per_step"], 4),
                                          "roofline": r3["roofline"], "slots": r3["info"].num_slots}
            ident = W.llama3_decode(seed=1001, identity_pages=True)
            r_id = decode_measure(ident, max(20, args.steps // 10), 5, peaks)
            secondary["page_permutation_overhead"] = {
                "identity_pages_ms": round(r_id["ms_per_step"], 4), "permuted_pages_ms": round(ms, 4),
                "overhead_pct": round((ms / r_id["ms_per_step"] - 1) * 100, 2)}
            del ident
            col = W.llama3_decode(seed=1001, page_size=1)
            r1 = decode_measure(col, max(20, args.steps // 10), 5, peaks)
            secondary["decode_page_size_1"] = {"value": round(r1["value"], 1), "unit": "GB/s",
                                               "ms_per_step": round(r1["ms_per_step"], 4), "roofline": r1["roofline"]}
            del col
            g8 = W.group8_decode(seed=1008)
            r8 = decode_measure(g8, max(20, args.steps // 10), 5, peaks,
                                kernel="prefill_kernel (group-8 decode on the tensor cores)")
            secondary["decode_group8"] = {"value": round(r8["value"], 1), "unit": "GB/s",
                                          "ms_per_step": round(r8["ms_per_step"], 4), "roofline": r8["roofline"],
                                          "workload": "64 q / 8 kv heads, head_dim 128, Llama-3-8B lengths"}
            del g8
            secondary["tiny_decode"] = tiny_measure(peaks)
            secondary["prefill"] = prefill_measure(peaks)
            secondary["cascade"] = cascade_measure(peaks)
            secondary["multilevel_cascade"] = multilevel_measure()
            secondary["append_rope"] = append_measure(peaks)
            secondary["tree_verify"] = tree_measure(peaks)
            secondary["mixed_batch"] = mixed_measure()
            secondary["prefill_page_size_1"] = prefill_measure(peaks, page_size=1)
            # The skewed batch again with the split turned off: each page list whole on
            # one warp, so the 131072-token request sets the step time.  Last, and any
            # error recorded in place: nothing after it uses the GPU.
            try:
                r4 = decode_measure(sk, max(20, args.steps // 10), 5, peaks, split_kv=False)
                secondary["skewed_decode"]["split_off"] = {
                    "value": round(r4["value"], 1), "unit": "GB/s", "ms_per_step": round(r4["ms_per_step"], 4),
                    "kernel_ms": round(r4["kernel_ms"], 4),
                    "split_speedup": round(r4["ms_per_step"] / r3["ms_per_step"], 2)}
            except Exception as e:
                secondary["skewed_decode"]["split_off"] = {"error": f"{type(e).__name__}: {e}"[:300]}
            del sk
    clocks.stop()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": b.batch, "num_qo_heads": 32, "num_kv_heads": 8, "head_dim": 128,
                   "page_size": 16, "kv_len": "U[512,4096]", "kv_bytes_per_step": b.kv_bytes(),
                   "l2": "inputs larger than L2 (KV read per step > 129 MB), no flush",
                   "step": "plan_run + decode kernel + merge kernel", "workers": info.workers,
                   "active_workers": info.active_workers, "split_sequences": info.num_merge},
        "hbm_frac_of_step": round(value / world / peaks["hbm_gbs"], 4),
        "roofline": res["roofline"],
        "host_plan": host_plan_entry(b),
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(b)
    if secondary:
        line["secondary"] = secondary
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_own(args)


if __name__ == "__main__":
    main()
