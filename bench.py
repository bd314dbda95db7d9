"""Benchmark of one PagedAttention step on GB300 (one JSON line on stdout).

Default workload: the mixed continuous-batch step (16 prompts of 1024 new
tokens with no past beside 240 decode sequences of one new token and past
lengths uniform 1024..8192, in a seeded random order; 32 query / 8 kv
heads, head_size 128, block_size 32, pool 20 % larger than needed with
shuffled blocks), seeded synthetic fp16 inputs: the largest of the five
workloads, and the one both halves of the metric are stated on.  A step is
one pa_forward: the prologue (device work list + paged cache write of the
new K/V rows), the tensor-core prefill of the prompts and, beside it on the
SMs the work list leaves, the split-KV decode with its combine.

--workload selects another step shape: `decode` (Llama-3-8B-shaped decode:
batch 64, past lengths uniform 512..4096, block_size 16), `long_window`
(Gemma-2-shaped window 4096 / softcap 50 decode), `rotary_decode`
(Llama-70B-shaped decode with rotary), `prefill` (16 prompts of 1024
tokens alone), `tiny`,
`decode_fp8` / `decode_int8` (the default decode step over an e4m3fn / int8
paged cache with per-channel scales; its K/V bytes count one byte per
element; `decode_fp8_bf16` / `decode_int8_bf16` the same with bfloat16
activations), `mla_decode` (DeepSeek-V3-shaped latent decode: 64 sequences,
128 heads, one 576-channel latent cache, block_size 64, past lengths
U{512..4096}; its K/V bytes are the latent rows, read once).

value    decode workloads: attended K/V bytes of the step / step time (GB/s),
         each admitted K and V element counted once per kv head; workloads
         with prompts: packed tokens of the step / step time (tokens/s).
e2e      the same metric through the C ABI with host inputs: pinned host
         Q/K/V, block table and lengths copied in and the output copied out
         inside the timed region; the paged pool is resident device state.
roofline the dominant kernel's algorithmic work over its own event-timed
         duration: decode = attended K/V + Q + output bytes of the decode
         sequences against the measured copy bandwidth; prefill = causal
         FLOPs 4 * D * H * sum(admitted keys) against the measured dense
         16-bit matmul rate (fp16 and bf16 share one nominal rate).
cpu_baseline  the fp64 CPU oracle on the host cores over a bounded sample of
         the same step's sequences.

--impl reference times the oracle alone (the pages ship no runnable
implementation; the oracle is the reference arm).  Under torchrun (N > 1)
each rank runs an independent replica on its own GPU ("replicas only":
the step has no cross-GPU exchange); value sums the ranks' work over the
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
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
def decode_rows(G):
    """Query rows of one decode item: q_len * G up to this goes to the decode
    kernel (its row tiles hold 8 rows; two tiles when G > 8)."""
    return 8 if G <= 8 else 16


# 8-bit cache variants of the Llama-3-8B-shaped decode step (per-channel
# scales, the quantized cache of the CUDA design, section 8)
QUANT_WORKLOADS = {"decode_fp8": 2, "decode_int8": 1, "decode_fp8_bf16": 2, "decode_int8_bf16": 1}
# bfloat16 activations and cache (the CUDA design registers the kernel for
# fp16 and bfloat16 activations, section 8.2) on the fp16 workloads' shapes
BF16_WORKLOADS = {"decode_bf16": "decode", "mixed_bf16": "mixed", "prefill_bf16": "prefill"}
CACHE_BF16 = 3


def quantized(step):
    return step.get("cache_dtype", 0) in (1, 2)


def act_bf16(step):
    """bfloat16 activations: a bfloat16 cache, or bfloat16 over 8-bit codes."""
    return step.get("cache_dtype", 0) == CACHE_BF16 or bool(step.get("act_bf16", False))


MLA_SCALE = 0.0723  # an explicit softmax scale (the latent width is not the model's head width)


def workload_shape(name):
    import torch

    import workloads
    index = {"tiny": 0, "decode": 1, "mixed": 2, "long_window": 3, "rotary_decode": 4}
    if name in QUANT_WORKLOADS:
        return workloads.config_shape(1)
    if name in BF16_WORKLOADS:
        return workload_shape(BF16_WORKLOADS[name])
    if name == "mla_decode":
        g = torch.Generator().manual_seed(3000 + 77)
        past = torch.randint(512, 4097, (64,), generator=g).tolist()
        return workloads.custom_shape("deepseek_v3_latent_decode_b64_h128_d576_dv512_bs64", 128, 1, 576, 64, past,
                                      [1] * 64, scale=MLA_SCALE, do_rotary=1, rotary_dim=64, seed=77)
    if name in index:
        return workloads.config_shape(index[name])
    if name == "prefill":
        return workloads.custom_shape("prefill_16x1024_h32_kv8_d128_bs32", 32, 8, 128, 32, [0] * 16,
                                      [1024] * 16, seed=2)
    raise ValueError(name)


def workload_options(name):
    """make_step keywords of a workload (8-bit cache variants)."""
    if name in QUANT_WORKLOADS:
        return dict(cache_dtype=QUANT_WORKLOADS[name], quant_type=2, act_bf16=name.endswith("_bf16"))
    if name in BF16_WORKLOADS:
        return dict(cache_dtype=CACHE_BF16)
    if name == "mla_decode":
        return dict(latent_v_head_size=512)
    return {}


def shape_name(name, shape):
    if name in BF16_WORKLOADS:
        return shape.name + "_bf16"
    if name in QUANT_WORKLOADS:
        tag = {2: "_e4m3_cache", 1: "_int8_cache"}[QUANT_WORKLOADS[name]]
        return shape.name + tag + ("_bf16" if name.endswith("_bf16") else "")
    return shape.name


def seq_lengths(step):
    past = step["past_sequence_lengths"].cpu().tolist()
    cum = step["cumulative_sequence_lengths"].cpu().tolist()
    return past, [cum[b + 1] - cum[b] for b in range(len(past))]


def admitted(pos, W):
    return min(pos + 1, W) if W >= 1 else pos + 1


def work_of(step, seqs=None):
    """Algorithmic work of (a subset of) the step's sequences."""
    past, q = seq_lengths(step)
    W, G = step["local_window_size"], step["num_heads"] // step["kv_num_heads"]
    Hk, H, D = step["kv_num_heads"], step["num_heads"], step["head_size"]
    eb = 1 if quantized(step) else 2  # bytes per cache element
    latent = step.get("kv_cache_layout", 0) == 1
    Dv = step.get("v_head_size") or D
    w = dict(kv_bytes=0, dec_kv_bytes=0, dec_qo_bytes=0, pre_flops=0, tokens=0, dec_flops=0)
    for b in (range(len(past)) if seqs is None else seqs):
        if q[b] == 0:
            continue
        L = past[b] + q[b]
        adm = min(L, W) if W >= 1 else L
        kv = adm * D * 2 if latent else adm * Hk * D * 2 * eb  # latent rows serve as K and V
        w["kv_bytes"] += kv
        w["tokens"] += q[b]
        if latent:
            w["dec_kv_bytes"] += kv
            w["dec_qo_bytes"] += q[b] * H * (D + Dv) * 2
            w["dec_flops"] += 2 * q[b] * H * adm * (D + Dv)
        elif q[b] * G <= decode_rows(G) or quantized(step):
            w["dec_kv_bytes"] += kv
            w["dec_qo_bytes"] += 2 * q[b] * H * D * 2
        else:
            w["pre_flops"] += 4 * D * H * sum(admitted(past[b] + j, W) for j in range(q[b]))
    return w


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def committed_traffic(kernel_file, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "paged_kv_cache_reshape_gb300", "csrc", kernel_file)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entries = json.load(f)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    for e in entries:
        if e.get("source") == kernel_file and e.get("source_sha256") == sha and e.get("workload") == workload:
            return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed loop runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = ""

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


def max_over_ranks(x, world, device="cpu"):
    """The slowest rank's time (all_reduce MAX); identity on one rank."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def metric_of(work, unit, seconds):
    return (work["kv_bytes"] / 1e9 if unit == "GB/s" else work["tokens"]) / seconds


def oracle_sample(step, budget_s, start_seq=0):
    """Runs the oracle's attention over whole sequences of the step from
    start_seq on (wrapping) until budget_s is spent.  Returns (seconds,
    sequences done, work of those sequences, next sequence, cores)."""
    import numpy as np

    import oracle

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    H, B = step["num_heads"], step["batch"]
    cum = step["cumulative_sequence_lengths"]
    if "_oracle_base" not in step:
        step["_oracle_base"] = oracle.forward(step, rows=np.zeros(0, dtype=np.int64))
    base = step["_oracle_base"]
    t0 = time.perf_counter()
    seqs = []
    b = start_seq
    while True:
        rows = np.arange(int(cum[b]) * H, int(cum[b + 1]) * H, dtype=np.int64)
        if rows.size and step.get("kv_cache_layout", 0) == 1:
            oracle.attention_latent(base["query_rot"], base["key_cache"], step["block_table"], cum,
                                    step["past_sequence_lengths"], H, step["head_size"], step["v_head_size"],
                                    step["block_size"], step["scale"], step["softcap"], step["local_window_size"],
                                    rows=rows, threads=cores)
        elif rows.size:
            oracle.attention(base["query_rot"], base["key_cache"], base["value_cache"], step["block_table"],
                             cum, step["past_sequence_lengths"], H, step["kv_num_heads"], step["head_size"],
                             step["block_size"], step["scale"], step["softcap"], step["local_window_size"],
                             rows=rows, threads=cores, cache_dtype=oracle.step_cache_dtype(step),
                             k_scale=step.get("k_scale"), v_scale=step.get("v_scale"),
                             per_channel=step.get("quant_type", 0) == 2, head_sink=step.get("head_sink"))
        seqs.append(b)
        b = (b + 1) % B
        if time.perf_counter() - t0 > budget_s or len(seqs) >= B:
            break
    return time.perf_counter() - t0, seqs, work_of(step, seqs), b, cores


def run_reference(args, rank, world):
    """The oracle as the reference arm: each of the W + K steps runs the
    oracle's attention over the next whole sequences of the same step, for a
    per-step time budget chosen so the run ends within a few minutes."""
    if rank != 0:
        return
    import workloads

    shape = workload_shape(args.workload)
    step = workloads.make_step(shape, device="cpu", **workload_options(args.workload))
    unit = "GB/s" if work_of(step)["pre_flops"] == 0 else "tokens/s"
    budget = min(args.ref_budget, max(0.02, 150.0 / (args.steps + args.warmup)))
    b, tot_t, done, cores = 0, 0.0, 0, 1
    acc = dict(kv_bytes=0, tokens=0)
    for i in range(args.warmup + args.steps):
        dt, seqs, w, b, cores = oracle_sample(step, budget, b)
        if i >= args.warmup:
            tot_t += dt
            done += len(seqs)
            acc["kv_bytes"] += w["kv_bytes"]
            acc["tokens"] += w["tokens"]
    value = metric_of(acc, unit, tot_t)
    sample = (f"{done} sequence-steps of the step's {step['batch']} sequences (all {step['num_heads']} "
              f"heads each), about {budget:.2f} s per step, {tot_t:.1f} s timed")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": shape_name(args.workload, shape), "sample": "bounded"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
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
    shape = workload_shape(args.workload)
    step = workloads.make_step(shape, device=dev, gen_device=str(dev), **workload_options(args.workload))
    host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in step.items()}
    work = work_of(host)
    unit = "tokens/s" if work["pre_flops"] > 0 else "GB/s"
    _, qlens = seq_lengths(host)
    # Replay-wide bound on query length (the op's attention_metadata): for a
    # decode step it lets the host skip launching the prefill kernel.
    op = pa.PagedAttention.for_step(step, max_query_len_bound=max(qlens))
    out_width = step["num_heads"] * (step.get("v_head_size") or step["head_size"])
    out = torch.empty(step["token_count"], out_width, device=dev,
                      dtype=torch.bfloat16 if act_bf16(step) else torch.float16)
    # A stream of the step's own (as a serving loop has): work on the legacy
    # default stream carries its implicit synchronisation with every other
    # blocking stream (measured: the decode step 104.4 us there, 98.9 us here).
    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    torch.cuda.set_stream(stream)
    sid = stream.cuda_stream

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # L2 flush between steps: a write of 2x L2, then a read of another 2x L2
    # buffer, so that the write-backs of the dirty lines the write leaves
    # finish before the step's events instead of inside the timed step.
    n_flush = max(2 * l2, 256 << 20) // 4
    flush_w = torch.empty(n_flush, dtype=torch.int32, device=dev)
    flush_r = torch.ones(n_flush, dtype=torch.int32, device=dev)
    flush_acc = torch.zeros((), dtype=torch.int64, device=dev)

    def flush_l2(i):
        flush_w.fill_(i)
        torch.sum(flush_r, dim=0, out=flush_acc)

    def fwd():
        op.forward(step, out, stream=sid)

    for _ in range(max(3, args.warmup)):
        flush_l2(1)
        fwd()
    torch.cuda.synchronize()
    assert op.device_error() == 0, "device error during warm-up"
    launches_per_step = op.last_launch_count()

    # ---- device-timed steps: one CUDA-graph replay of pa_forward each (the
    # step is capture-safe: no host sync, no allocation); L2 flushed before
    # each replay, outside the events.  A second graph, captured with the
    # library's per-kernel events on, times the kernels alone.
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

    def timed_loop(fn, n, sample_kernels):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ker = {pa.PA_STAGE_DECODE: [], pa.PA_STAGE_PREFILL: []}
        for i in range(n):
            flush_l2(i)
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
            if sample_kernels and (i % 16 == 15 or i == n - 1):
                for s in ker:
                    v = op.kernel_time_ms(s)
                    if v >= 0:
                        ker[s].append(v)
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)], ker

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        # Soak: the same replays (L2 flushed between them) for at least one
        # second before the timed loop, so the clock samples see the GPU
        # under this load; the timed loop follows at once.
        t_soak = time.perf_counter()
        n_soak = 0
        while time.perf_counter() - t_soak < args.soak_s:
            for i in range(32):
                flush_l2(i)
                run()
            n_soak += 32
            torch.cuda.synchronize()
        soak_s = time.perf_counter() - t_soak
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t_wall0 = time.perf_counter()
        step_ms, _ = timed_loop(run, args.steps, False)
        t_wall = time.perf_counter() - t_wall0
        op.set_option(pa.PA_OPT_KERNEL_TIMING, 1)
        _, ker_ms = timed_loop(run_timed, min(args.steps, 256), True)
        op.set_option(pa.PA_OPT_KERNEL_TIMING, 0)
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)
    value = world * metric_of(work, unit, ms * 1e-3)

    hbm, tflops, peak_kind = measured_peaks()
    rooflines = {}
    if ker_ms[pa.PA_STAGE_DECODE] and work["dec_kv_bytes"]:
        t = statistics.mean(ker_ms[pa.PA_STAGE_DECODE])
        alg = work["dec_kv_bytes"] + work["dec_qo_bytes"]
        ct = {0: "", 1: ", int8", 2: ", e4m3", 3: ", bf16"}[host.get("cache_dtype", 0)]
        if quantized(host) and act_bf16(host):
            ct += ", bf16 out"
        latent = host.get("kv_cache_layout", 0) == 1
        latent_tc = latent and shape.num_heads % 128 == 0  # the tcgen05 latent kernel serves these
        kname = (("mla_tc_kernel" if latent_tc else "mla_decode_kernel") if latent
                 else f"decode_kernel<{shape.head_size}{ct}>")
        if work["dec_flops"]:
            ach = work["dec_flops"] / (t * 1e-3) / 1e12
            rooflines["decode_tensor"] = {
                "bound": "tensor", "kernel": kname, "achieved": ach, "peak": tflops,
                "peak_kind": f"{peak_kind} bf16 matmul burst (the kernel runs "
                             + ("tcgen05 kind::f16 MMAs)" if latent_tc else "m16n8k16 fp16 HMMA)"),
                "unit": "TFLOP/s", "frac": ach / tflops, "traffic": None,
                "algorithmic_flops_per_launch": work["dec_flops"], "launch_ms": t - 1e-9}
        rooflines["decode"] = {
            "bound": "hbm", "kernel": kname, "achieved": alg / (t * 1e-3) / 1e9,
            "peak": hbm, "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s",
            "frac": alg / (t * 1e-3) / 1e9 / hbm,
            "traffic": committed_traffic(("mla_tc.cu" if latent_tc else "mla.cu") if latent else "decode.cu",
                                         shape_name(args.workload, shape)),
            "algorithmic_bytes_per_launch": alg,
            "launch_ms": t}
    if ker_ms[pa.PA_STAGE_PREFILL] and work["pre_flops"]:
        t = statistics.mean(ker_ms[pa.PA_STAGE_PREFILL])
        ach = work["pre_flops"] / (t * 1e-3) / 1e12
        # head_size 64/128 run the two-tile kernel, 256 the one-tile kernel
        pair = shape.head_size <= 128
        bf = ", bf16" if act_bf16(host) else ""
        rooflines["prefill"] = {
            "bound": "tensor",
            "kernel": (f"prefill_pair_kernel<{shape.head_size}{bf}>" if pair
                       else f"prefill_kernel<{shape.head_size}{bf}>"),
            "achieved": ach, "peak": tflops,
            "peak_kind": f"{peak_kind} bf16 matmul burst; fp16 has the same nominal dense rate",
            "unit": "TFLOP/s", "frac": ach / tflops,
            "traffic": committed_traffic("prefill_pair.cu" if pair else "prefill.cu", shape_name(args.workload, shape)),
            "algorithmic_flops_per_launch": work["pre_flops"], "launch_ms": t}
    dominant = max(rooflines, key=lambda k: rooflines[k]["launch_ms"]) if rooflines else None

    # ---- end to end through the C ABI with host buffers
    names = [n for n in ("query", "key", "value", "block_table", "cumulative_sequence_lengths",
                         "past_sequence_lengths") if step.get(n) is not None]
    pinned = {n: step[n].cpu().pin_memory() for n in names}
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = out_host.numel() * out_host.element_size()
    e_steps = max(10, min(args.steps, 500))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(e_steps)]
    for i in range(e_steps + 3):
        flush_l2(i)
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
    e2e_ms = max_over_ranks(statistics.mean(s.elapsed_time(e) for s, e in zip(es, ee)), world, dev)
    e2e = world * metric_of(work, unit, e2e_ms * 1e-3)
    assert op.device_error() == 0, "device error in the timed region"

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if host.get("cache_dtype", 0) == CACHE_BF16 else "f16",
        "data": "synthetic",
        "config": {"workload": shape_name(args.workload, shape), "batch": shape.batch,
                   "token_count": shape.token_count,
                   "num_heads": shape.num_heads, "kv_num_heads": shape.kv_num_heads,
                   "head_size": shape.head_size, "block_size": shape.block_size,
                   "attended_kv_bytes_per_step": work["kv_bytes"], "prefill_flops_per_step": work["pre_flops"],
                   "l2": "flushed before every step (write of 2x L2, then read of another 2x L2), outside the "
                         "step's events",
                   "launch": ("eager" if args.eager else "cuda_graph replay of one pa_forward") + " on a dedicated stream",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": rooflines.get(dominant),
        "gpu_launches": launches_per_step * (args.steps + min(args.steps, 256)),
        "gpu_launches_per_step": launches_per_step,
        "e2e": {"value": e2e, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "clocks": dict(clk.summary(), soak_s=soak_s, soak_steps=n_soak,
                       sampled="every 100 ms over a soak of the same replays and the timed loop"),
        "wall_s_timed_region": t_wall,
    }
    if unit == "GB/s":
        line["pct_of_8tbs_hbm"] = 100.0 * value / world / NOMINAL_HBM_GBS
    else:
        # a step with prompts: its attended K/V bytes over the whole step time
        kv_gbs = work["kv_bytes"] / (ms * 1e-3) / 1e9
        line["step_attended_kv_gbs"] = kv_gbs
        line["step_attended_kv_pct_of_8tbs_hbm"] = 100.0 * kv_gbs / NOMINAL_HBM_GBS
    for k, r in rooflines.items():
        if k != dominant:
            line[f"roofline_{k}"] = r
    if not args.no_cpu_baseline:
        dt, seqs, w, _, cores = oracle_sample(host, args.ref_budget)
        sample = (f"attention of {len(seqs)} of {host['batch']} sequences (all {host['num_heads']} heads each) "
                  f"of the step, {dt:.1f} s")
        line["cpu_baseline"] = {"value": metric_of(w, unit, dt), "unit": unit, "cores": cores, "kind": "oracle",
                                "sample": sample}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed",
                    choices=["decode", "mixed", "long_window", "rotary_decode", "prefill", "tiny"]
                    + sorted(QUANT_WORKLOADS) + sorted(BF16_WORKLOADS) + ["mla_decode"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch pa_forward directly instead of a graph replay")
    ap.add_argument("--soak-s", type=float, default=1.5, help="seconds of untimed replays under the clock sampler")
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
