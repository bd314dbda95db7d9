"""Benchmark of one PagedAttention step on GB300 (one JSON line on stdout).

Workload: the Llama-3-8B-shaped decode step (batch 64, 32 query / 8 kv
heads, head_size 128, block_size 16, one new token per sequence, past
lengths uniform 512..4096, pool 20 % larger than needed with shuffled
blocks), seeded synthetic fp16 inputs.  A step is one pa_forward: the
work-list build, the paged cache write of the 64 new K/V rows and the
split-KV attention with its combine.

value   = attended K/V bytes of the step / device time of the step (GB/s);
          attended bytes = sum_b admitted_b * kv_heads * head_size * 2 (K, V)
          * 2 bytes, each KV element counted once per step.
e2e     = the same metric through the C ABI with host inputs: pinned host
          Q/K/V, block table and lengths copied in and the output copied out
          inside the timed region; the paged pool is resident device state.
roofline= the decode kernel's algorithmic bytes (attended K/V + Q + output)
          over its own event-timed duration, against the measured copy
          bandwidth.
cpu_baseline = the fp64 CPU oracle on the host cores over a bounded sample
          of the same step's sequences.

--impl reference times the oracle alone (the pages ship no runnable
implementation; the oracle is the reference arm).  Under torchrun (N > 1)
each rank runs an independent replica on its own GPU ("replicas only":
the step has no cross-GPU exchange); value sums the ranks' bytes over the
slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attended-KV GB/s (% of 8 TB/s HBM); mixed-batch tokens/s"
UNIT = "GB/s"
WORKLOAD_INDEX = 1
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def attended_kv_bytes(step) -> int:
    """Bytes of K and V the step must read: per sequence the keys its last
    token admits (min(L_b, W) under a window), per kv head, K and V, fp16."""
    past = step["past_sequence_lengths"].cpu().tolist()
    cum = step["cumulative_sequence_lengths"].cpu().tolist()
    W = step["local_window_size"]
    keys = 0
    for b, p in enumerate(past):
        q = cum[b + 1] - cum[b]
        if q:
            L = p + q
            keys += min(L, W) if W >= 1 else L
    return keys * step["kv_num_heads"] * step["head_size"] * 2 * 2


def seq_kv_bytes(step, b) -> int:
    past = int(step["past_sequence_lengths"][b])
    cum = step["cumulative_sequence_lengths"]
    q = int(cum[b + 1] - cum[b])
    W = step["local_window_size"]
    L = past + q
    adm = (min(L, W) if W >= 1 else L) if q else 0
    return adm * step["kv_num_heads"] * step["head_size"] * 4


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def decode_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, or None
    when the decode kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    src = os.path.join(ROOT, "paged_kv_cache_reshape_gb300", "csrc", "decode.cu")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if d.get("decode_cu_sha256") != sha or d.get("workload") != "llama3_8b_decode_b64_h32_kv8_d128_bs16":
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed loop runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.out = out
        else:
            self.out = ""

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(step_host, budget_s=12.0):
    """The oracle (as it stands) on the host cores, over whole sequences of the
    step until the time budget is spent.  Returns (GB/s, cores, sample text)."""
    import numpy as np

    import oracle

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    H = step_host["num_heads"]
    cum = step_host["cumulative_sequence_lengths"]
    B = step_host["batch"]
    # Rotary / cache write of the whole step first (part of the oracle's step).
    base = oracle.forward(step_host, rows=np.zeros(0, dtype=np.int64))
    t0 = time.perf_counter()
    done, nbytes = 0, 0
    for b in range(B):
        rows = np.arange(int(cum[b]) * H, int(cum[b + 1]) * H, dtype=np.int64)
        if rows.size:
            oracle.attention(base["query_rot"], base["key_cache"], base["value_cache"],
                             step_host["block_table"], cum, step_host["past_sequence_lengths"], H,
                             step_host["kv_num_heads"], step_host["head_size"],
                             step_host["block_size"], step_host["scale"], step_host["softcap"],
                             step_host["local_window_size"], rows=rows, threads=cores)
        nbytes += seq_kv_bytes(step_host, b)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    sample = (f"attention of {done} of {B} sequences (all {H} heads each) of the step, "
              f"{dt:.1f} s, {nbytes / 1e6:.1f} MB attended K/V")
    return nbytes / dt / 1e9, cores, sample


def run_reference(args, rank, world):
    """The oracle as the reference arm: each of the W + K steps runs the
    oracle's attention over the next whole sequences of the same step, for a
    per-step time budget chosen so the run ends within a few minutes."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    import workloads

    shape = workloads.config_shape(WORKLOAD_INDEX)
    step = workloads.make_step(shape, device="cpu")
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    H, B = step["num_heads"], step["batch"]
    cum = step["cumulative_sequence_lengths"]
    base = oracle.forward(step, rows=np.zeros(0, dtype=np.int64))
    budget = min(args.ref_budget, max(0.02, 150.0 / (args.steps + args.warmup)))
    b = 0
    tot_bytes, tot_t, seqs = 0, 0.0, 0
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        nbytes = 0
        while True:
            rows = np.arange(int(cum[b]) * H, int(cum[b + 1]) * H, dtype=np.int64)
            oracle.attention(base["query_rot"], base["key_cache"], base["value_cache"],
                             step["block_table"], cum, step["past_sequence_lengths"], H,
                             step["kv_num_heads"], step["head_size"], step["block_size"],
                             step["scale"], step["softcap"], step["local_window_size"], rows=rows,
                             threads=cores)
            nbytes += seq_kv_bytes(step, b)
            b = (b + 1) % B
            if i >= args.warmup:
                seqs += 1
            if time.perf_counter() - t0 > budget:
                break
        if i >= args.warmup:
            tot_bytes += nbytes
            tot_t += time.perf_counter() - t0
    value = tot_bytes / tot_t / 1e9
    sample = (f"{seqs} sequence-steps of the step's 64 sequences (all {H} heads each), "
              f"about {budget:.2f} s per step, {tot_t:.1f} s timed")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": shape.name, "sample": "bounded"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch

    import paged_kv_cache_reshape_gb300 as pa
    import workloads
    from paged_kv_cache_reshape_gb300 import builder

    builder.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    shape = workloads.config_shape(WORKLOAD_INDEX)
    step = workloads.make_step(shape, device=dev, gen_device=str(dev))
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in step.items()}
    kv_bytes = attended_kv_bytes(host)
    T, H, D = step["token_count"], step["num_heads"], step["head_size"]
    decode_alg_bytes = kv_bytes + 2 * T * H * D * 2  # + Q read + output write

    op = pa.PagedAttention.for_step(step)
    out = torch.empty_like(step["query"])
    stream = torch.cuda.current_stream(dev)
    sid = stream.cuda_stream

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)

    def fwd():
        op.forward(step, out, stream=sid)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        fwd()
    torch.cuda.synchronize()
    assert op.device_error() == 0, "device error during warm-up"
    launches_per_step = op.last_launch_count()

    # ---- device-timed steps: one CUDA-graph replay of pa_forward each (the
    # step is capture-safe: no host sync, no allocation); L2 flushed before
    # each replay, outside the events.  A second graph, captured with the
    # library's per-kernel events on, times the decode kernel alone.
    def capture():
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            op.forward(step, out, stream=cap.cuda_stream)
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        return g

    run = fwd if args.eager else capture().replay
    op.set_option(pa.PA_OPT_KERNEL_TIMING, 1)
    run_timed = fwd if args.eager else capture().replay
    op.set_option(pa.PA_OPT_KERNEL_TIMING, 0)

    def timed_loop(fn, n, sample_decode):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        dec = []
        for i in range(n):
            flush.fill_(i)
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
            if sample_decode and (i % 16 == 15 or i == n - 1):
                dec.append(op.kernel_time_ms(pa.PA_STAGE_DECODE))
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)], dec

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t_wall0 = time.perf_counter()
        step_ms, _ = timed_loop(run, args.steps, False)
        t_wall = time.perf_counter() - t_wall0
        op.set_option(pa.PA_OPT_KERNEL_TIMING, 1)
        _, dec_ms = timed_loop(run_timed, min(args.steps, 256), True)
        op.set_option(pa.PA_OPT_KERNEL_TIMING, 0)
    if world > 1:
        torch.distributed.barrier()
    ms = statistics.mean(step_ms)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    value = world * kv_bytes / (ms * 1e-3) / 1e9

    # ---- decode kernel alone: events around it inside pa_forward, same stream
    dec = statistics.mean(dec_ms)
    peak, peak_kind = measured_peaks()
    achieved = decode_alg_bytes / (dec * 1e-3) / 1e9
    traffic = decode_traffic()

    # ---- end to end through the C ABI with host buffers
    names = ["query", "key", "value", "block_table", "cumulative_sequence_lengths", "past_sequence_lengths"]
    pinned = {n: step[n].cpu().pin_memory() for n in names}
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = out_host.numel() * out_host.element_size()
    e_steps = max(10, args.steps // 4)
    es = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps)]
    for i in range(e_steps + 3):
        flush.fill_(i)
        k = i - 3
        if k >= 0:
            es[k].record(stream)
        for n in names:
            step[n].copy_(pinned[n], non_blocking=True)
        fwd()
        out_host.copy_(out, non_blocking=True)
        if k >= 0:
            ee[k].record(stream)
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(es, ee))
    if world > 1:
        t = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e = world * kv_bytes / (e2e_ms * 1e-3) / 1e9
    assert op.device_error() == 0, "device error in the timed region"

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "pct_of_8tbs_hbm": 100.0 * value / world / NOMINAL_HBM_GBS,
        "config": {"workload": shape.name, "batch": shape.batch, "num_heads": shape.num_heads,
                   "kv_num_heads": shape.kv_num_heads, "head_size": shape.head_size,
                   "block_size": shape.block_size, "attended_kv_bytes_per_step": kv_bytes,
                   "l2": "flushed before every step (write of 2x L2), outside the step's events",
                   "launch": "eager" if args.eager else "cuda_graph replay of one pa_forward",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "kernel": "decode_kernel<128>", "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes_per_launch": decode_alg_bytes,
                     "launch_ms": dec},
        "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": launches_per_step * (args.steps + min(args.steps, 256)),
        "clocks": clk.summary(),
        "wall_s_timed_region": t_wall,
    }
    if not args.no_cpu_baseline:
        v, cores, sample = cpu_baseline(host, budget_s=args.ref_budget)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch pa_forward directly instead of a graph replay")
    ap.add_argument("--ref-budget", type=float, default=12.0, help="seconds of oracle work per sample")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
