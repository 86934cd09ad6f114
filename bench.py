#!/usr/bin/env python3
"""Benchmark of the fused exp-normalised GQA attention path on GB300.

One step = one ``mg_attn_run`` (the fused partial kernel plus, when the N axis is split, the
combine kernel) over one batch of the GQA tutorial workload: Q (2,256,64), K (2,64,4096),
V (2,4096,64) fp16, Q,K ~ U(-0.5,0.5), V ~ N(0,1), seed 0 (Mirage documentation,
tutorials/group-query-attention, "Define GQA Computation Graph").

Timing follows the method the Mirage docs describe for candidate kernels (warm-up runs,
then CUDA events around a long run of back-to-back calls, time / calls), on one stream,
with these additions:
  * every step reads a different input/output buffer set; the sets together are more than
    twice the L2 size, so each call reads its inputs from HBM, not L2;
  * the timed steps are replayed from a CUDA graph (host launch cost excluded); a plain
    stream loop is timed too and reported beside it;
  * the roofline fraction uses the fused kernel's average duration: the timed region / K
    when a step is that one kernel, else events the library records around each launch;
  * two floors outside the roofline formula are measured in the same run and reported
    beside it (``ceilings``): the launch floor of the plan's launch shape and the time of the
    B*M*N exponentials at the measured per-SM rate;
  * the end-to-end number runs the host-buffer entry point: host->device copies of Q, K, V,
    the kernels, and the device->host copy of O, every step.
The CPU baseline is the fp64 oracle (test infrastructure) on the host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Multi-GPU: one process per GPU under torch.distributed.run; every rank runs its own
independent replica (the path needs no exchange), value = all ranks' FLOPs / max time.
"""

from __future__ import annotations

import argparse
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

METRIC = "fused GQA muGraph TFLOP/s and µs/call at 1 GB300; % of roofline"
WORKLOAD = "gqa"  # Q (2,256,64), K (2,64,4096), V (2,4096,64)
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "mg_attn_fwd_partial_gqa.md")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
QUEUE_FILL_CYCLES = 2_000_000  # device-side sleep ahead of a timed region (~1 ms at 2 GHz)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample length")
    ap.add_argument("--per-config-steps", type=int, default=2000, help="graph-replayed calls per workload")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-workload table")
    return ap.parse_args()


def workload_shape():
    from attention_mugraph_gb300 import inputs

    B, M, N, d, a = inputs.CONFIGS[WORKLOAD]
    return B, M, N, d, a


def flops_per_step(B, M, N, d):
    return 4.0 * B * M * N * d


def bytes_per_step(B, M, N, d):
    return 2.0 * (B * M * d + B * d * N + B * N * d + B * M * d)


def load_peaks():
    if os.path.exists(PEAKS_PATH):
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def ceilings(info, B, M, N, exp_rate_ns, roof_us):
    """The two floors outside the roofline formula, for one plan: the launch floor of its launch
    shape (a no-work kernel with the fused kernel's prologue, measured now) and the time of its
    B*M*N exponentials at the measured per-SM rate on every SM."""
    import attention_mugraph_gb300 as mg

    floor = mg.diag_launch_floor(info["grid_ctas"], max(1, info["cluster_ctas"]), info["smem_bytes"], True, 1000)
    t_exp = B * M * N / (exp_rate_ns * info["num_sms"]) / 1e3
    return {"launch_floor_us": floor, "exp_time_us": t_exp, "roofline_us": roof_us,
            "floor_us": max(floor, t_exp, roof_us)}


def source_code_text(text: str) -> str:
    """C++ source without its comments and blank lines: what a digest of the code should see."""
    import re

    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


FUSED_SOURCES = ("attention_mugraph_gb300/csrc/mg_attn_kernels.cuh", "attention_mugraph_gb300/csrc/ptx.cuh")
FEW_ROW_SOURCES = ("attention_mugraph_gb300/csrc/mg_attn_swap.cuh",) + FUSED_SOURCES


def kernel_source_digest(sources=FUSED_SOURCES):
    """Digest of a kernel's code (by default the fused kernel's two headers; FEW_ROW_SOURCES for
    the few-row kernel; comments left out), recorded beside the ncu counters in the committed
    summary; a change of code invalidates the recorded traffic."""
    import hashlib

    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(source_code_text(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the fused kernel from the committed ncu summary, if it was taken
    on the current kernel source (its digest line matches); else None."""
    if not os.path.exists(TRAFFIC_PATH):
        return None
    fields = {}
    with open(TRAFFIC_PATH) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_digest") != kernel_source_digest():
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's elapsed time (all_reduce MAX); the identity on one rank."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps (weak scaling), timed by the slowest."""
    return flops_per_step * world * steps / (max_ms * 1e-3) / 1e12


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, smax, loaded, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            try:
                if len(parts) > 9 and float(parts[9]) >= 50.0:
                    loaded.append(sm[-1])
            except ValueError:
                pass
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(loaded or sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "samples_under_load": len(loaded),
                "sm_mhz_median_all": statistics.median(sm)}


# ------------------------------------------------------------------ CPU (oracle) timing

def time_oracle(q, k, v, seconds: float, rows_per_call=None, threads=None):
    """Run the fp64 oracle repeatedly for about `seconds`; returns (calls, elapsed, rows, threads).
    rows_per_call=None runs the whole workload per call, else that many leading rows; threads=None
    uses every host thread OpenMP offers."""
    import oracle

    lib = oracle.load_library()
    threads = oracle.max_threads(lib) if threads is None else int(threads)
    B, M, d = q.shape
    rows = list(range(B * M if rows_per_call is None else min(rows_per_call, B * M)))
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.attention_rows(q, k, v, rows, threads=threads, lib=lib)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return calls, el, len(rows), threads


def cpu_baseline(q, k, v, seconds):
    B, M, N, d = q.shape[0], q.shape[1], k.shape[2], q.shape[2]
    calls, el, rows, threads = time_oracle(q, k, v, seconds)
    fl = 4.0 * rows * N * d * calls
    # The same oracle on one thread, on a sample of leading rows (a third of the time budget).
    c1, el1, rows1, _ = time_oracle(q, k, v, max(1.0, seconds / 3), rows_per_call=32, threads=1)
    fl1 = 4.0 * rows1 * N * d * c1
    return {"value": fl / el / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{calls} full oracle evaluations of the {WORKLOAD} workload ({rows} rows x N={N} x d={d}, "
                      f"fp64) in {el:.1f} s on {threads} host threads",
            "single_thread": {"value": fl1 / el1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                              "sample": f"{c1} evaluations of the first {rows1} rows in {el1:.1f} s on 1 thread"}}


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle, timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import torch

    from attention_mugraph_gb300 import inputs

    B, M, N, d, a = workload_shape()
    q, k, v = inputs.make_inputs(B, M, N, d, a, seed=0)
    import oracle

    lib = oracle.load_library()
    threads = oracle.max_threads(lib)
    # Size each step's sample (leading rows of the workload) so the whole run takes ~2 minutes.
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, list(range(B * M)), threads=threads, lib=lib)
    per_row = (time.perf_counter() - t0) / (B * M)
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows_per_step = int(max(1, min(B * M, budget / max(per_row, 1e-9))))
    rows = list(range(rows_per_step))
    for _ in range(args.warmup):
        oracle.attention_rows(q, k, v, rows, threads=threads, lib=lib)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_rows(q, k, v, rows, threads=threads, lib=lib)
    el = time.perf_counter() - t0
    fl = 4.0 * rows_per_step * N * d * args.steps
    value = fl / el / 1e12
    sample = (f"each step: the first {rows_per_step} of {B * M} rows of the {WORKLOAD} workload "
              f"(N={N}, d={d}) in fp64 on {threads} host threads")
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(B, M, N, d, a, extra={"arm": "fp64 CPU oracle"}),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    del torch


def workload_config(B, M, N, d, a, extra=None):
    cfg = {"workload": f"GQA tutorial graph: Q ({B},{M},{d}), K ({B},{d},{N}), V ({B},{N},{d}) fp16",
           "B": B, "M": M, "N": N, "d": d, "inputs": f"Q,K ~ U(-{a},{a}), V ~ N(0,1), seed 0"}
    if extra:
        cfg.update(extra)
    return cfg


# ------------------------------------------------------------------ GPU arm

def measure_workload(name, steps, peaks, stream, exp_rate_ns, flags=0):
    """Graph-replayed µs/call over rotating buffer sets (> 2x L2) and the fused kernel's own time for
    one named workload; returns a dict for the JSON line's per_config field."""
    import torch

    import attention_mugraph_gb300 as mg
    from attention_mugraph_gb300 import inputs

    B, M, N, d, a = inputs.CONFIGS[name]
    fl = flops_per_step(B, M, N, d)
    by = bytes_per_step(B, M, N, d)
    q, k, v = inputs.make_inputs(B, M, N, d, a, seed=0)
    l2 = int(getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "L2_cache_size", 0)
             or 132 * 1024 * 1024)
    n_sets = max(2, math.ceil(2 * l2 / by))
    dev = [(q.cuda(), k.cuda(), v.cuda(), torch.empty((B, M, d), dtype=torch.float16, device="cuda"))
           for _ in range(n_sets)]
    plan = mg.Plan(B, M, N, d, flags=flags)
    ptrs = [tuple(t.data_ptr() for t in s) for s in dev]
    sh = stream.cuda_stream
    with torch.cuda.stream(stream):
        for i in range(max(3, n_sets)):
            plan.run_ptr(*ptrs[i % n_sets], stream=sh)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        g.capture_begin()
        for i in range(n_sets):
            plan.run_ptr(*ptrs[i], stream=sh)
        g.capture_end()
    reps = max(1, steps // n_sets)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(QUEUE_FILL_CYCLES)  # the GPU waits while the host queues the replays
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    e1.record(stream)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * n_sets)
    # Fused kernel alone (library-recorded events, host queue fed ahead of the GPU).
    nk = min(200, max(n_sets, 20))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nk)]
    for pair in evs:
        for ev in pair:
            ev.record(stream)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(20_000_000)
        for i in range(nk):
            plan.set_timing_events(*evs[i])
            plan.run_ptr(*ptrs[i % n_sets], stream=sh)
    plan.set_timing_events(None, None)
    stream.synchronize()
    k_us = statistics.median([b.elapsed_time(e) for b, e in evs]) * 1e3
    t_tensor = fl / (peaks["bf16_tflops"] * 1e12)
    t_hbm = by / (peaks["hbm_gbs"] * 1e9)
    roof = max(t_tensor, t_hbm) * 1e6
    st = plan.status()
    info = plan.info
    if st != mg.MG_OK:
        raise SystemExit(f"{name}: device status {st}")
    plan.destroy()
    return {"B": B, "M": M, "N": N, "d": d, "us_per_call": us, "tflops": fl / (us * 1e-6) / 1e12,
            "hbm_gbs": by / (us * 1e-6) / 1e9, "roofline_us": roof, "roofline_frac": roof / us,
            "bound": "hbm" if t_hbm >= t_tensor else "tensor", "fused_kernel_us_median": k_us,
            "n_split": info["n_split"], "cluster_ctas": info["cluster_ctas"], "buffer_sets": n_sets,
            "ceilings": ceilings(info, B, M, N, exp_rate_ns, roof)}


def per_config_summary(line):
    """Compact table as the line's last key: for every workload, [µs per call, % of roofline] of the
    graph as written and of the two opt-in variants, plus the headline step."""
    out = {"gqa_headline": [round(line["us_per_call"], 3), round(100 * line["roofline_fraction_of_step"], 2)]}
    for key, tag in (("per_config", "plain"), ("per_config_safe_softmax", "safe_softmax"),
                     ("per_config_qk_norm", "qk_norm")):
        if key in line:
            out[tag] = {name: [round(r["us_per_call"], 2), round(100 * r["roofline_frac"], 1)]
                        for name, r in line[key].items()}
    out["format"] = "[us per call, % of roofline]"
    return out


def main():
    args = parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist

    import attention_mugraph_gb300 as mg
    from attention_mugraph_gb300 import build, inputs

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if world > 1:
            dist.barrier()

    build.build()
    B, M, N, d, a = workload_shape()
    fl = flops_per_step(B, M, N, d)
    alg_bytes = bytes_per_step(B, M, N, d)

    q, k, v = inputs.make_inputs(B, M, N, d, a, seed=0)
    props = torch.cuda.get_device_properties(local_rank)
    l2 = int(getattr(props, "L2_cache_size", 0) or 132 * 1024 * 1024)
    set_bytes = int(alg_bytes)
    n_sets = max(2, math.ceil(2 * l2 / set_bytes))
    Qs = [q.cuda() for _ in range(n_sets)]
    Ks = [k.cuda() for _ in range(n_sets)]
    Vs = [v.cuda() for _ in range(n_sets)]
    Os = [torch.empty((B, M, d), dtype=torch.float16, device="cuda") for _ in range(n_sets)]
    ptrs = [(Qs[i].data_ptr(), Ks[i].data_ptr(), Vs[i].data_ptr(), Os[i].data_ptr()) for i in range(n_sets)]

    plan = mg.Plan(B, M, N, d)
    info = plan.info
    stream = torch.cuda.Stream()
    # Clocks are sampled over the whole GPU arm (warm-up, the timed regions, the per-workload
    # tables): the headline region alone is shorter than one 200 ms sample.
    arm_clocks = ClockSampler(local_rank).__enter__()
    sh = stream.cuda_stream

    def step(i):
        plan.run_ptr(*ptrs[i % n_sets], stream=sh)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()

    # Graphs: one covers a whole rotation of buffer sets; a second covers the remainder.
    def capture(count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            g.capture_begin()
            for i in range(count):
                step(i)
            g.capture_end()
        return g

    full, rem = divmod(args.steps, n_sets)
    g_full = capture(n_sets) if full else None
    g_rem = capture(rem) if rem else None
    for _ in range(3):  # graph warm-up
        if g_full:
            g_full.replay()
        if g_rem:
            g_rem.replay()
    stream.synchronize()

    def timed(fn):
        barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        # The stream sleeps on the device (~1 ms) before the first event, so that the host has
        # queued the timed launches by the time the GPU reaches it: the events then time the
        # GPU's execution of the K steps, not the host's submission of the first of them.
        with torch.cuda.stream(stream):
            torch.cuda._sleep(QUEUE_FILL_CYCLES)
        ev0.record(stream)
        fn()
        ev1.record(stream)
        ev1.synchronize()
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(ev0.elapsed_time(ev1), world, device="cuda")

    def graph_steps():
        with torch.cuda.stream(stream):
            for _ in range(full):
                g_full.replay()
            if g_rem:
                g_rem.replay()

    # Timed region 1 (the value): K steps replayed from CUDA graphs.
    ms_graph = timed(graph_steps)

    # Timed region 2: the same K steps as a plain host loop of mg_attn_run calls.
    def loop_steps():
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                step(i)

    ms_loop = timed(loop_steps)

    # Fused kernel alone: events recorded by the library around it. Each batch of launches is
    # queued behind a device-side sleep so the host runs ahead and the events time the GPU, not
    # the Python launch loop.
    batch = 100
    n_k = max(batch, (min(args.steps, max(n_sets, 1000)) // batch) * batch)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_k)]
    for pair in evs:  # torch creates the CUDA event on its first record; the library re-records it
        for ev in pair:
            ev.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for b0 in range(0, n_k, batch):
            torch.cuda._sleep(20_000_000)  # ~10 ms of GPU time while the host queues the batch
            for i in range(b0, b0 + batch):
                plan.set_timing_events(*evs[i])
                step(i)
    plan.set_timing_events(None, None)
    stream.synchronize()
    k_ms = [b.elapsed_time(e) for b, e in evs]
    fwd_us = statistics.mean(k_ms) * 1e3
    fwd_us_median = statistics.median(k_ms) * 1e3

    # End to end through the host-buffer entry point (pinned host memory), every step copying
    # Q, K, V in and O out. Consecutive calls overlap (each call's inputs cross the host link while
    # the previous call computes), so at least 200 calls are timed: with a handful, the first
    # call's unoverlapped start would weigh on the mean.
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    ho = torch.empty((B, M, d), dtype=torch.float16).pin_memory()
    n_e2e = min(max(args.steps, 200), 2000)
    with torch.cuda.stream(stream):
        for _ in range(3):
            plan.run_host(hq, hk, hv, ho, stream=stream)
    stream.synchronize()

    def e2e_steps():
        with torch.cuda.stream(stream):
            for _ in range(n_e2e):
                plan.run_host(hq, hk, hv, ho, stream=stream)

    ms_e2e = timed(e2e_steps)
    h2d = int(q.numel() + k.numel() + v.numel()) * 2
    d2h = int(ho.numel()) * 2

    st = plan.status()
    if st != mg.MG_OK:
        raise SystemExit(f"device status {st} after the bench")

    peaks, peak_kind = load_peaks()
    t_tensor = fl / (peaks["bf16_tflops"] * 1e12)
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    bound = "hbm" if t_hbm >= t_tensor else "tensor"
    # The fused kernel's average launch duration. When a step is that one kernel, the timed
    # region itself (CUDA events on the launching stream around K back-to-back launches) gives it;
    # events recorded around each single launch would add their own latency to a few-µs kernel
    # and end the overlap of consecutive launches (a launch that starts early runs beside the one
    # before it), so that figure is reported beside as the launch timed alone.
    # With a second (combine) kernel per step, the per-launch events bracket the fused kernel.
    if info["kernels_per_run"] == 1:
        dur_us = ms_graph * 1e3 / args.steps
        dur_source = ("timed region / steps (one kernel per step; consecutive launches overlap, so "
                      "this is the time each launch adds to the sequence)")
    else:
        dur_us = fwd_us
        dur_source = "mean of CUDA events recorded around each fused-kernel launch"
    if bound == "hbm":
        achieved = alg_bytes / (dur_us * 1e-6) / 1e9
        peak = peaks["hbm_gbs"]
        unit = "GB/s"
    else:
        achieved = fl / (dur_us * 1e-6) / 1e12
        peak = peaks["bf16_tflops"]
        unit = "TFLOP/s"

    # Exponential rate of the fused kernel's instruction sequence (MUFU), and of the FMA-pipe
    # polynomial it can move columns to, per SM clock and per SM ns.
    exp_clk, exp_ns = mg.diag_exp_rate(2000, poly=False)
    poly_clk, poly_ns = mg.diag_exp_rate(2000, poly=True)

    if rank != 0:
        arm_clocks.__exit__(None, None, None)
        plan.destroy()
        if world > 1:
            dist.destroy_process_group()
        return
    us_graph = ms_graph * 1e3 / args.steps
    us_loop = ms_loop * 1e3 / args.steps
    value = job_tflops(fl, args.steps, world, ms_graph)
    roof_t = max(t_tensor, t_hbm)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_graph / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": workload_config(B, M, N, d, a, extra={
            "l2": (f"inputs larger than L2: {n_sets} rotating Q/K/V/O buffer sets of {set_bytes} B "
                   f"({n_sets * set_bytes / 2**20:.0f} MiB, > 2x the {l2 / 2**20:.0f} MiB L2); each step "
                   f"reads a set untouched for {n_sets - 1} steps"),
            "launch": "CUDA graph replay of back-to-back mg_attn_run calls on one stream",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "n_split": info["n_split"], "grid_ctas": info["grid_ctas"], "stages": info["stages"],
            "kernels_per_step": info["kernels_per_run"]}),
        "us_per_call": us_graph,
        "roofline_time_us": roof_t * 1e6,
        "roofline_fraction_of_step": roof_t * 1e6 / us_graph,
        "stream_loop": {"us_per_call": us_loop, "value": job_tflops(fl, args.steps, world, ms_loop),
                        "unit": "TFLOP/s"},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                     "traffic": recorded_traffic(), "kernel": "mg_attn_fwd_partial",
                     "kernel_us": dur_us, "kernel_us_source": dur_source,
                     "event_bracketed_us_mean": fwd_us, "event_bracketed_us_median": fwd_us_median,
                     "algorithmic_bytes_per_launch": alg_bytes, "flops_per_launch": fl,
                     "peak_source": f"{peak_kind}: MEASURED_PEAKS.json "
                                    f"{'hbm_gbs' if bound == 'hbm' else 'bf16_tflops'} (burst)",
                     "tensor_frac": fl / (dur_us * 1e-6) / 1e12 / peaks["bf16_tflops"]},
        "e2e": {"value": job_tflops(fl, n_e2e, world, ms_e2e), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": n_e2e, "us_per_call": ms_e2e * 1e3 / n_e2e},
        "gpu_launches": args.steps * info["kernels_per_run"],
        "ceilings": dict(ceilings(info, B, M, N, exp_ns, roof_t * 1e6),
                         exp_per_clk_per_sm_mufu=exp_clk, exp_per_ns_per_sm_mufu=exp_ns,
                         exp_per_clk_per_sm_fma_poly=poly_clk, exp_per_ns_per_sm_fma_poly=poly_ns),
    }
    if world == 1:
        if not args.no_per_config:
            from attention_mugraph_gb300 import inputs as _inputs

            line["per_config"] = {name: measure_workload(name, args.per_config_steps, peaks, stream, exp_ns)
                                  for name in _inputs.CONFIG_ORDER}
            # The max-subtracted variant (MG_FLAG_SAFE_SOFTMAX) on the same workloads.
            line["per_config_safe_softmax"] = {
                name: measure_workload(name, args.per_config_steps, peaks, stream, exp_ns, flags=mg.MG_FLAG_SAFE_SOFTMAX)
                for name in _inputs.CONFIG_ORDER}
            # QK-norm attention (MG_FLAG_QK_NORM, which implies the max-subtracted evaluation).
            line["per_config_qk_norm"] = {
                name: measure_workload(name, args.per_config_steps, peaks, stream, exp_ns, flags=mg.MG_FLAG_QK_NORM)
                for name in _inputs.CONFIG_ORDER}
    arm_clocks.__exit__(None, None, None)
    line["clocks"] = dict(arm_clocks.summary(), window="the whole GPU arm: warm-up, timed regions, "
                                                      "per-workload tables")
    if world == 1:
        line["cpu_baseline"] = cpu_baseline(q, k, v, args.cpu_seconds)
        line["summary"] = per_config_summary(line)
    print(json.dumps(line), flush=True)
    plan.destroy()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
