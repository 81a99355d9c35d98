#!/usr/bin/env python3
"""Benchmark: packed varlen attention with modality-tagged 3D RoPE on GB300.

One step = one pass of the hot path over one packed request: continuation time shift + tagged
RoPE of Q and K (h3_rope_apply) and block-diagonal attention over cu_seqlens
(h3_varlen_attn_fwd).  Default workload: the H3-shaped request of 58,758 tokens (text 558 +
audio 200 + video 29x40x50), 40 heads x 128, bf16, segments [0,558,758,58758], capacity 58,816
with NaN pad rows.  Metric: attention TFLOP/s = 4*H*D*sum(n_g^2) / step time.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU fp64 oracle instead (the only
reference that exists for this method): on a bounded sample of the H3 request or of the window
layer pair, or in full for the worked example and the 4,096-token request.
"""
from __future__ import annotations

import argparse
import json
import os
import resource
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "packed varlen attn TFLOP/s @58,758 tok, 40x128 bf16; % GB300 dense BF16 peak"
UNIT = "TFLOP/s"


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workloads' short measurements after the headline")
    p.add_argument("--config-steps", type=int, default=5,
                   help="timed steps of each other workload measured after the headline")
    p.add_argument("--workload", default="h3_full_request",
                   choices=["h3_full_request", "single_request_4k", "continuation_batch",
                            "continuation_batch_4seg",
                            "video_segment_16k", "window_grid", "window_grid_16x24x84",
                            "vsa_video", "vsa_video_16x24x84", "vsa_video_shared_half", "continuation_window",
                            "tiny_example"],
                   help="h3_full_request is the metric's workload; the others are side measurements")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return dict(hbm_gbs=float(j["hbm_gbs"]), bf16_tflops=float(j["bf16_tflops"]),
                    bf16_tflops_sustained=float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------------------------------------
# replicas: every rank runs the same workload (weak scaling); the job time is the slowest rank's
# ------------------------------------------------------------------------------------------------
def max_over_ranks(ms: float, world: int, device=None) -> float:
    """Slowest rank's time (no-op for one rank); works on any process-group backend."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(work_per_rank: float, world: int, job_ms: float) -> float:
    """Whole-job TFLOP/s: the work of all replicas over the slowest replica's time."""
    return world * work_per_rank / (job_ms / 1e3) / 1e12


# ------------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.reader = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            try:
                power.append(float(parts[3]))
            except ValueError:
                power.append(float("nan"))
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        # samples under load: power draw at least half of the highest seen in the window
        pw = np.array(power, dtype=np.float64)
        loaded = [c for c, w in zip(sm, pw) if np.isfinite(w) and w >= 0.5 * np.nanmax(pw)] if sm else []
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "sm_mhz_loaded": float(np.median(loaded)) if loaded else None,
                "power_w_max": float(np.nanmax(pw)) if sm else None,
                "reasons": sorted(reasons), "samples": len(sm), "samples_loaded": len(loaded)}


# ------------------------------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ------------------------------------------------------------------------------------------------
def oracle_sample_step(wl, rows):
    """One sampled oracle step on the host cores.

    The fp64 oracle rotates the sampled query rows and every key of their segment, then computes
    attention for those rows.  The job-equivalent time charges the keys' RoPE pro rata (it is
    shared by all rows of the segment in a full pass).  Returns
    (attention flops, job-equivalent seconds, threads used, wall seconds).
    """
    import oracle

    g = int(np.searchsorted(wl.cu_seqlens, rows[0], side="right")) - 1
    a, b = int(wl.cu_seqlens[g]), int(wl.cu_seqlens[g + 1])
    assert np.all((rows >= a) & (rows < b))
    ru0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    ko = oracle.rope_apply(wl.k, wl.pos, wl.tag, wl.cu_requests, wl.start_frames, rows=np.arange(a, b))
    t1 = time.perf_counter()
    qo = oracle.rope_apply(wl.q, wl.pos, wl.tag, wl.cu_requests, wl.start_frames, rows=rows)
    vo = wl.v[a:b].double().numpy()
    q_seg = np.zeros((b - a, wl.num_heads, wl.head_dim))
    q_seg[rows - a] = qo
    oracle.varlen_attention(q_seg, ko, vo, [0, b - a], rows=rows - a)
    t2 = time.perf_counter()
    ru1 = resource.getrusage(resource.RUSAGE_SELF)
    cpu = (ru1.ru_utime - ru0.ru_utime) + (ru1.ru_stime - ru0.ru_stime)
    flops = 4.0 * wl.num_heads * wl.head_dim * (b - a) * len(rows)
    job_s = (t2 - t1) + (t1 - t0) * len(rows) / (b - a)
    return flops, job_s, max(1, round(cpu / (t2 - t0))), t2 - t0


def sample_rows(wl, n_rows, seed):
    g = int(np.argmax(np.diff(wl.cu_seqlens)))  # the long video segment
    a, b = int(wl.cu_seqlens[g]), int(wl.cu_seqlens[g + 1])
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(np.arange(a, b), size=min(n_rows, b - a), replace=False))


def cpu_baseline(wl, n_rows=512):
    """The oracle on the host cores on a bounded sample (about 10-30 s); TFLOP/s."""
    f, job_s, threads, wall = oracle_sample_step(wl, sample_rows(wl, n_rows, 1))
    return {"value": f / job_s / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n_rows} query rows of the 58,000-row video segment x 40 heads: fp64 RoPE of those "
                      f"rows and of all 58,000 keys (charged pro rata), then fp64 attention; "
                      f"{f / 1e12:.3f} TFLOP, {wall:.1f} s wall; host has "
                      f"{len(os.sched_getaffinity(0))} cores"}


def _cpu_threads(ru0, ru1, wall):
    cpu = (ru1.ru_utime - ru0.ru_utime) + (ru1.ru_stime - ru0.ru_stime)
    return max(1, round(cpu / wall)) if wall > 0 else 1


def _reference_line(args, metric, value, unit, higher, ms, config, threads, sample):
    return {"metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": higher, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference", "config": config,
            "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def _reference_full_packed(args):
    """The oracle's whole pass (fp64 RoPE of Q and K, then attention over every row) each step:
    the worked example and the 4,096-token request are small enough to time in full."""
    import oracle
    import workloads

    wl = workloads.WORKLOADS[args.workload]()
    times, threads = [], 1
    for i in range(args.warmup + args.steps):
        ru0, t0 = resource.getrusage(resource.RUSAGE_SELF), time.perf_counter()
        qr = oracle.rope_apply(wl.q, wl.pos, wl.tag, wl.cu_requests, wl.start_frames)
        kr = oracle.rope_apply(wl.k, wl.pos, wl.tag, wl.cu_requests, wl.start_frames)
        oracle.varlen_attention(qr, kr, wl.v, wl.cu_seqlens)
        t1, ru1 = time.perf_counter(), resource.getrusage(resource.RUSAGE_SELF)
        if i >= args.warmup:
            times.append(t1 - t0)
            threads = _cpu_threads(ru0, ru1, t1 - t0)
    sec = float(np.mean(times))
    config = {"workload": wl.name, "tokens": wl.num_tokens, "heads": wl.num_heads, "head_dim": wl.head_dim,
              "cu_seqlens": [int(x) for x in wl.cu_seqlens]}
    sample = "the whole pass each step: fp64 RoPE of Q and K, then fp64 attention over every row"
    if args.workload == "tiny_example":
        line = _reference_line(args, "worked-example step latency (RoPE + varlen attention, 45 tokens)",
                               sec * 1e6, "us", False, sec * 1e3, config, threads, sample)
    else:
        line = _reference_line(args, f"packed varlen attn TFLOP/s ({wl.name})",
                               wl.attention_flops() / sec / 1e12, UNIT, True, sec * 1e3, config, threads,
                               sample)
    print(json.dumps(line), flush=True)


def _reference_window(args, windows_per_layer=4):
    """Both window layers of the 32x48x84 grid on a sample: each step draws windows of each layer
    uniformly at random, packs their rows, runs fp64 attention and restores them; each layer's
    time is scaled to the whole layer by its window count (an unbiased estimate of the whole
    layer's time; one full layer takes minutes here)."""
    import oracle
    from workloads import window_grid

    wl = window_grid()
    H, D = wl.num_heads, wl.head_dim
    shifts = [wl.shift if sh else (0, 0, 0) for sh in wl.layer_shifted]
    total_flops = 0.0
    parts = []
    for sh in shifts:
        perm, cu = oracle.window_partition(wl.grid, wl.window, sh)
        sizes = np.diff(cu).astype(np.float64)
        parts.append((perm, cu, sizes))
        total_flops += 4.0 * H * D * float(np.sum(sizes ** 2))
    out = np.zeros((wl.num_tokens, H, D))  # the layer's output in grid order (allocated once)
    times, threads = [], 1
    for i in range(args.warmup + args.steps):
        rng = np.random.default_rng(500 + i)
        job = 0.0
        for (perm, cu, sizes), (q, k, v) in zip(parts, wl.layers):
            pick = np.sort(rng.choice(sizes.size, windows_per_layer, replace=False))
            ru0, t0 = resource.getrusage(resource.RUSAGE_SELF), time.perf_counter()
            rows = np.concatenate([perm[cu[w]:cu[w + 1]] for w in pick])
            sub_cu = np.concatenate([[0], np.cumsum(sizes[pick])]).astype(np.int64)
            qp, kp, vp = (oracle.window_pack(x, rows) for x in (q, k, v))
            o, _ = oracle.varlen_attention(qp, kp, vp, sub_cu)
            out[rows] = o
            t1, ru1 = time.perf_counter(), resource.getrusage(resource.RUSAGE_SELF)
            threads = _cpu_threads(ru0, ru1, t1 - t0)
            job += (t1 - t0) * sizes.size / windows_per_layer
        if i >= args.warmup:
            times.append(job)
    sec = float(np.mean(times))
    config = {"workload": wl.name, "tokens": wl.num_tokens, "heads": H, "head_dim": D,
              "windows_sampled_per_layer": windows_per_layer}
    sample = (f"per step {windows_per_layer} windows of each layer drawn uniformly: fp64 pack, attention and "
              "restore of their rows, each layer's time scaled by its window count")
    print(json.dumps(_reference_line(args, "shifted 3D window attention TFLOP/s (2 layers, attention in place "
                                     "on the grid)", total_flops / sec / 1e12, UNIT, True, sec * 1e3, config,
                                     threads, sample)), flush=True)


def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.workload in ("tiny_example", "single_request_4k"):
        return _reference_full_packed(args)
    if args.workload == "window_grid":
        return _reference_window(args)
    if args.workload != "h3_full_request":
        print(json.dumps({"impl": "reference", "unavailable": "the oracle is timed on h3_full_request, "
                          "single_request_4k, tiny_example and window_grid only"}), flush=True)
        return
    from workloads import h3_full_request

    wl = h3_full_request()
    n_rows = 96
    times, flops, threads = [], 0.0, 1
    for i in range(args.warmup + args.steps):
        f, job_s, th, _ = oracle_sample_step(wl, sample_rows(wl, n_rows, 100 + i))
        if i >= args.warmup:
            times.append(job_s)
            flops, threads = f, th
    ms = 1e3 * float(np.mean(times))
    value = flops / (ms / 1e3) / 1e12
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": wl.name, "tokens": wl.num_tokens, "heads": wl.num_heads,
                       "head_dim": wl.head_dim, "cu_seqlens": [int(x) for x in wl.cu_seqlens],
                       "sample_rows_per_step": n_rows},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"per step {n_rows} query rows of the video segment x 40 heads: "
                                       "fp64 RoPE of those rows and of all 58,000 keys (charged pro "
                                       "rata), then fp64 attention"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------
# dense bf16 tcgen05 work per SM per cycle: one 128 x 128 x 16 MMA (524,288 FLOP) every 64 cycles
# (measured on this GPU with a sequence of such MMAs issued back to back)
TENSOR_FLOP_PER_SM_CYCLE = 8192.0


def run_ours(args, rank, world, local_rank):
    import packed_varlen_attention_modality_gb300 as h3

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    h3.load_library()
    peaks = load_peaks()
    if args.workload.startswith("window_grid"):
        line = run_window(args, rank, world, dev, h3, peaks)
    elif args.workload.startswith("vsa_video"):
        line = run_vsa(args, rank, world, dev, h3, peaks)
    elif args.workload == "continuation_window":
        line = run_continuation(args, rank, world, dev, h3, peaks)
    elif args.workload == "tiny_example":
        line = run_latency(args, rank, world, dev, h3)
    else:
        line = run_packed(args, rank, world, dev, h3, peaks)
    if args.workload == "h3_full_request" and not args.no_configs:
        if world == 1:
            line["configs"] = collect_configs(args, rank, world, dev, h3, peaks)
        else:
            line["configs"] = {"skipped": "the other workloads are measured at one GPU only"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_packed(args, rank, world, dev, h3, peaks, wl=None):
    """One packed request per step: tagged RoPE of Q and K (with the continuation shift), then
    block-diagonal attention over cu_seqlens.  The headline workload also gets the end-to-end leg
    and the CPU baseline."""
    import workloads

    headline = args.workload == "h3_full_request"
    if wl is None:
        wl = workloads.WORKLOADS[args.workload]()
    H, D, C, N = wl.num_heads, wl.head_dim, wl.capacity, wl.num_tokens
    flops = wl.attention_flops()

    q, k, v = (t.to(dev) for t in (wl.q, wl.k, wl.v))
    pos = torch.from_numpy(wl.pos).to(dev)
    tag = torch.from_numpy(wl.tag).to(dev)
    cu = torch.from_numpy(wl.cu_seqlens).to(dev)
    cu_req = torch.from_numpy(wl.cu_requests).to(dev)
    frames = torch.from_numpy(wl.start_frames).to(dev)
    qr, kr, o = torch.empty_like(q), torch.empty_like(k), torch.empty_like(q)
    lse = torch.empty((H, C), dtype=torch.float32, device=dev)
    max_seqlen = wl.max_seqlen
    ws = torch.empty(max(16, h3.varlen_attn_workspace_size(wl.num_segments, H, max_seqlen, D)),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        h3.rope_apply(q, k, pos, tag, cu_req, frames, num_tokens=N, q_out=qr, k_out=kr)
        if ev is not None:
            ev[1].record(stream)
        h3.varlen_attn_fwd(qr, kr, v, cu, max_seqlen, out=o, lse=lse, workspace=ws)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if h3.get_device_error(dev) != 0:
        raise RuntimeError("device error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    if h3.get_device_error(dev) != 0:
        raise RuntimeError("device error during the timed steps")
    rope_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    attn_each = [e[1].elapsed_time(e[2]) for e in evs]
    attn_ms = float(np.mean(attn_each))
    ms_per_step = total_ms / args.steps
    value = job_throughput(flops, world, ms_per_step)

    attn_tflops = flops / (attn_ms / 1e3) / 1e12
    rope_bytes = 4.0 * N * H * D * 2 + 13.0 * N  # read+write Q and K (bf16) + pos (12 B) + tag (1 B)
    rope_gbs = rope_bytes / (rope_ms / 1e3) / 1e9
    traffic = None
    traffic_file = os.path.join(ROOT, "profiles", "attn_fwd_dram_traffic.json")
    if headline and os.path.exists(traffic_file):
        with open(traffic_file) as f:
            tj = json.load(f)
        if tj.get("kernel_source_sha") == _kernel_sha():
            traffic = tj.get("dram_bytes_per_launch")
    # tensor peak at the clock the kernel actually ran at (sampled, never set): SMs x per-SM rate
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # (only when at least three samples fell under load: a timed region shorter than about a
    # second gives the 200 ms sampler nothing to go on)
    mhz = clocks.get("sm_mhz_loaded") if (clocks.get("samples_loaded") or 0) >= 3 else None
    clock_peak = sms * TENSOR_FLOP_PER_SM_CYCLE * mhz * 1e6 / 1e12 if mhz else None

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if headline and not args.no_e2e:
        e2e = run_e2e(args, world, dev, h3, wl, q, k, v, pos, tag, cu, cu_req, frames, flops, max_seqlen, ws)

    cpu = None
    if headline and rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)

    return {
        "metric": METRIC if headline else f"packed varlen attn TFLOP/s ({wl.name})", "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "tokens": N, "capacity": C, "heads": H, "head_dim": D,
                   "cu_seqlens": [int(x) for x in wl.cu_seqlens], "attention_flop": flops,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2 (each of Q, K, V, O is %.0f MB > 129 MB)"
                         % (C * H * D * 2 / 1e6)},
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": attn_tflops / peaks["bf16_tflops"],
                     "traffic": traffic, "kernel": "attn_fwd_kernel<%d>" % D,
                     "peak_source": peaks["source"] + " bf16_tflops (burst)",
                     "frac_of_sustained": attn_tflops / peaks["bf16_tflops_sustained"],
                     "attn_ms": attn_ms,
                     "peak_at_sampled_clock": clock_peak,
                     "frac_at_sampled_clock": attn_tflops / clock_peak if clock_peak else None,
                     "sampled_clock_basis": "%d SMs x %d FLOP/cycle (128x128x16 bf16 MMA per 64 "
                                            "cycles) x median SM MHz under load" % (sms, TENSOR_FLOP_PER_SM_CYCLE)},
        "kernels": {"rope": {"ms": rope_ms, "gbs": rope_gbs, "bytes": rope_bytes,
                             "frac_hbm": rope_gbs / peaks["hbm_gbs"]},
                    "attn_fwd": {"ms": attn_ms, "tflops": attn_tflops,
                                 "ms_median": float(np.median(attn_each)),
                                 "ms_min": float(np.min(attn_each)),
                                 "tflops_median": flops / (float(np.median(attn_each)) / 1e3) / 1e12}},
        "clocks": clocks,
        # RoPE, attention plan, attention per step, and the merge of split items when the workspace
        # holds the split area (segments of 1,024 rows or more)
        "gpu_launches": (4 if max_seqlen >= 1024 else 3) * args.steps,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }


def collect_configs(args, rank, world, dev, h3, peaks):
    """Short timed measurements of the other workloads, each against its own bound, after
    the headline: the 4,096-token request and the 4-request continuation batch (tensor), the
    window layer pair in place and through pack/attention/unpack (HBM), block-sparse attention
    at top 1/8 (useful and issued tensor work), the continuation window's row movement (HBM) and
    the worked example's latency.  Few steps each, so the whole run stays within minutes."""
    import workloads

    def sub(name):
        return argparse.Namespace(**{**vars(args), "workload": name, "steps": max(1, args.config_steps),
                                     "warmup": 3, "no_e2e": True, "no_cpu_baseline": True})

    def packed(line):
        at, ro = line["kernels"]["attn_fwd"], line["kernels"]["rope"]
        return {"workload": line["config"]["workload"], "segments": len(line["config"]["cu_seqlens"]) - 1,
                "bound": "tensor", "attn_ms": at["ms"], "attn_ms_median": at["ms_median"],
                "attn_tflops": at["tflops"], "frac": at["tflops"] / peaks["bf16_tflops"],
                "frac_of_sustained": at["tflops"] / peaks["bf16_tflops_sustained"],
                "frac_at_sampled_clock": line["roofline"]["frac_at_sampled_clock"],
                "rope_ms": ro["ms"], "rope_frac_hbm": ro["frac_hbm"],
                "sm_mhz_loaded": line["clocks"].get("sm_mhz_loaded")}

    out = {"steps_each": max(1, args.config_steps), "warmup_each": 3,
           "peaks": {"bf16_tflops": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"],
                     "source": peaks["source"]}}
    t0 = time.time()
    out["single_request_4k"] = packed(run_packed(sub("single_request_4k"), rank, world, dev, h3, peaks))
    torch.cuda.empty_cache()
    wl = workloads.continuation_batch()
    out["continuation_batch"] = packed(run_packed(sub("continuation_batch"), rank, world, dev, h3, peaks, wl))
    torch.cuda.empty_cache()
    wl.cu_seqlens = np.asarray(wl.cu_requests, dtype=np.int32)  # one segment per request
    wl.name = "continuation_4req_4seg_40x128"
    out["continuation_batch_4seg"] = packed(run_packed(sub("continuation_batch_4seg"), rank, world, dev, h3,
                                                       peaks, wl))
    del wl
    torch.cuda.empty_cache()

    w = run_window(sub("window_grid"), rank, world, dev, h3, peaks)
    out["window_grid"] = {"workload": w["config"]["workload"], "bound": "hbm",
                          "in_place_roofline": w["roofline"], "layers": w["layers"],
                          "in_place_ms_per_layer_pair": w["ms_per_step"],
                          "packed_ms_per_layer_pair": w["packed_path"]["ms_per_step"]}
    torch.cuda.empty_cache()
    vs = run_vsa(sub("vsa_video"), rank, world, dev, h3, peaks)
    ka = vs["kernels"]["attn"]
    out["vsa_video"] = {"workload": vs["config"]["workload"], "bound": "tensor",
                        "select_ms": vs["kernels"]["select"]["ms"], "attn_ms": ka["ms"],
                        "tflops_useful": ka["tflops_useful"], "frac_useful": ka["tflops_useful"] / peaks["bf16_tflops"],
                        "tflops_executed": ka["tflops_executed"],
                        "frac_executed": ka["tflops_executed"] / peaks["bf16_tflops"],
                        "executed_over_useful": ka["tflops_executed"] / ka["tflops_useful"],
                        "shared_selection_frac": ka["shared_selection_frac"], "steps": ka["steps"],
                        "steps_unshared": ka["steps_unshared"]}
    torch.cuda.empty_cache()
    cw = run_continuation(sub("continuation_window"), rank, world, dev, h3, peaks)
    out["continuation_window"] = {"workload": cw["config"]["workload"], "bound": "hbm",
                                  **{k: {"ms": v["ms"], "gbs": v["gbs"], "frac_hbm": v["frac_hbm"]}
                                     for k, v in cw["kernels"].items()}}
    torch.cuda.empty_cache()
    lat = run_latency(sub("tiny_example"), rank, world, dev, h3)
    out["tiny_example"] = {"workload": lat["config"]["workload"], "bound": "launch latency",
                           **lat["latency_us"]}
    out["wall_s"] = time.time() - t0
    return out


def run_e2e(args, world, dev, h3, wl, q, k, v, pos, tag, cu, cu_req, frames, flops, max_seqlen, ws):
    """End-to-end throughput through the public API: every step copies its inputs from pinned host
    memory, runs RoPE + attention and reads the output back to pinned host memory.  The steps run
    as a double-buffered pipeline on three streams (host->device, compute, device->host), so step
    i's copies overlap the compute of its neighbours, as a server streaming requests would."""
    N = wl.num_tokens
    host = {name: t.cpu().pin_memory() for name, t in
            (("q", q), ("k", k), ("v", v), ("pos", pos), ("tag", tag), ("cu", cu),
             ("cu_req", cu_req), ("frames", frames))}
    bi = sum(t.numel() * t.element_size() for t in host.values())
    nbuf = 2
    bufs = [{name: torch.empty_like(t, device=dev) for name, t in host.items()} for _ in range(nbuf)]
    outs = [torch.empty_like(q) for _ in range(nbuf)]
    host_out = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(nbuf)]
    bo = host_out[0].numel() * host_out[0].element_size()
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    s_h2d, s_cmp, s_d2h = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event(enable_timing=False)
    h2d_done = [ev() for _ in range(nbuf)]
    cmp_done = [ev() for _ in range(nbuf)]
    d2h_done = [ev() for _ in range(nbuf)]

    def e2e_step(i):
        b = i % nbuf
        d = bufs[b]
        with torch.cuda.stream(s_h2d):
            if i >= nbuf:
                s_h2d.wait_event(cmp_done[b])  # buffer b's inputs were consumed by step i - 2
            for name, t in host.items():
                d[name].copy_(t, non_blocking=True)
            h2d_done[b].record(s_h2d)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(h2d_done[b])
            if i >= nbuf:
                s_cmp.wait_event(d2h_done[b])  # outs[b] was read back by step i - 2
            h3.rope_apply(d["q"], d["k"], d["pos"], d["tag"], d["cu_req"], d["frames"], num_tokens=N,
                          q_out=qr, k_out=kr)
            h3.varlen_attn_fwd(qr, kr, d["v"], d["cu"], max_seqlen, out=outs[b], workspace=ws)
            cmp_done[b].record(s_cmp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(cmp_done[b])
            host_out[b].copy_(outs[b], non_blocking=True)
            d2h_done[b].record(s_d2h)

    for i in range(nbuf):  # warm-up of the copy paths
        e2e_step(i)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    # 20 steps at least: the pipeline's fill (first copy in) and drain (last copy out), ~12 ms on
    # the H3 request, are then a small share of the timed region
    n_e2e = max(20, args.steps)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(s_h2d)
    for i in range(n_e2e):
        e2e_step(i)
    s1.record(s_d2h)  # after the last read-back, which follows every earlier operation
    torch.cuda.synchronize(dev)
    e_ms = max_over_ranks(s0.elapsed_time(s1) / n_e2e, world, dev)
    if h3.get_device_error(dev) != 0:
        raise RuntimeError("device error during the end-to-end steps")
    return {"value": job_throughput(flops, world, e_ms), "unit": UNIT, "h2d_bytes_per_step": int(bi),
            "d2h_bytes_per_step": int(bo), "ms_per_step": e_ms, "steps": n_e2e,
            "pipeline": "double-buffered: host->device, compute and device->host on three streams"}


def run_window(args, rank, world, dev, h3, peaks):
    """Shifted 3D window attention (32x48x84 grid, 4x8x8 windows, shift 2,4,4; 24 x 128): per step,
    for each of the two layers (unshifted, shifted): window pack of Q/K/V -> varlen attention
    over the window segments -> restore original order."""
    from workloads import window_grid

    # window_grid_16x24x84: a quarter of the grid (198 MB per tensor, still larger than L2), small
    # enough for a full ncu capture
    wl = window_grid(grid=(16, 24, 84)) if args.workload == "window_grid_16x24x84" else window_grid()
    n, H, D = wl.num_tokens, wl.num_heads, wl.head_dim
    layers = [tuple(t.to(dev) for t in lay) for lay in wl.layers]
    shifts = [wl.shift if sh else (0, 0, 0) for sh in wl.layer_shifted]
    nwins = [h3.window_count(wl.grid, wl.window, s) for s in shifts]
    perms = [torch.empty(n, dtype=torch.int32, device=dev) for _ in shifts]
    cus = [torch.empty(nw + 1, dtype=torch.int32, device=dev) for nw in nwins]
    packed = [torch.empty_like(layers[0][0]) for _ in range(3)]
    op = torch.empty_like(layers[0][0])
    wss = [torch.empty(h3.varlen_attn_workspace_size(nw, H, 256, D), dtype=torch.uint8, device=dev)
           for nw in nwins]
    outs = [torch.empty_like(layers[0][0]) for _ in layers]
    stream = torch.cuda.current_stream(dev)

    # attention FLOPs per layer from the partition sizes (closed form per axis)
    def axis_sizes(L, w, s):
        return [min(L, (i + 1) * w - s) - max(0, i * w - s) for i in range((L + s + w - 1) // w)]
    flops = []
    for s in shifts:
        sq = [sum(e * e for e in axis_sizes(L, w, sh)) for L, w, sh in zip(wl.grid, wl.window, s)]
        flops.append(4.0 * H * D * sq[0] * sq[1] * sq[2])

    def step(ev=None):
        for li, (q, k, v) in enumerate(layers):
            if ev is not None:
                ev[li][0].record(stream)
            h3.window_pack(wl.grid, wl.window, shifts[li], [q, k, v], perm=perms[li], cu_seqlens=cus[li],
                           outs=packed)
            if ev is not None:
                ev[li][1].record(stream)
            h3.varlen_attn_fwd(packed[0], packed[1], packed[2], cus[li], 256, out=op, workspace=wss[li])
            if ev is not None:
                ev[li][2].record(stream)
            h3.window_unpack(perms[li], op, outs[li])
            if ev is not None:
                ev[li][3].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if h3.get_device_error(dev) != 0:
        raise RuntimeError("device error during warm-up")
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in layers] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    ms_per_step = t0.elapsed_time(t1) / args.steps
    per = {}
    row = H * D * 2
    pack_bytes = 2.0 * 3 * n * row + 4.0 * n   # read + write Q, K, V rows; perm
    unpack_bytes = 2.0 * n * row + 4.0 * n
    attn_bytes = 4.0 * n * row                   # Q, K, V read once, O written once
    for li in range(len(layers)):
        tp = float(np.mean([e[li][0].elapsed_time(e[li][1]) for e in evs]))
        ta = float(np.mean([e[li][1].elapsed_time(e[li][2]) for e in evs]))
        tu = float(np.mean([e[li][2].elapsed_time(e[li][3]) for e in evs]))
        name = "shifted" if wl.layer_shifted[li] else "regular"
        per[name] = {"windows": nwins[li],
                     "pack": {"ms": tp, "gbs": pack_bytes / tp / 1e6, "frac_hbm": pack_bytes / tp / 1e6 / peaks["hbm_gbs"]},
                     "attn": {"ms": ta, "tflops": flops[li] / ta / 1e9, "gbs": attn_bytes / ta / 1e6,
                              "frac_hbm": attn_bytes / ta / 1e6 / peaks["hbm_gbs"],
                              "hbm_roofline_ms": max(attn_bytes / peaks["hbm_gbs"] / 1e6,
                                                     flops[li] / peaks["bf16_tflops"] / 1e9)},
                     "unpack": {"ms": tu, "gbs": unpack_bytes / tu / 1e6,
                                "frac_hbm": unpack_bytes / tu / 1e6 / peaks["hbm_gbs"]}}
    # the same two layers with attention read and written in place on the grid (no packed copies)
    fouts = [torch.empty_like(layers[0][0]) for _ in layers]

    def fused_step(ev=None):
        for li, (q, k, v) in enumerate(layers):
            if ev is not None:
                ev[li][0].record(stream)
            h3.window_attn_fwd(q, k, v, wl.grid, wl.window, shifts[li], out=fouts[li])
            if ev is not None:
                ev[li][1].record(stream)

    for _ in range(max(3, args.warmup)):
        fused_step()
    torch.cuda.synchronize(dev)
    fevs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in layers] for _ in range(args.steps)]
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(args.steps):
        fused_step(fevs[i])
    f1.record(stream)
    torch.cuda.synchronize(dev)
    if h3.get_device_error(dev) != 0:
        raise RuntimeError("device error during the in-place window steps")
    fused_ms_per_step = max_over_ranks(f0.elapsed_time(f1) / args.steps, world, dev)
    for li in range(len(layers)):
        tf = float(np.mean([e[li][0].elapsed_time(e[li][1]) for e in fevs]))
        name = "shifted" if wl.layer_shifted[li] else "regular"
        per[name]["in_place_attn"] = {
            "ms": tf, "tflops": flops[li] / tf / 1e9, "gbs": attn_bytes / tf / 1e6,
            "frac_hbm": attn_bytes / tf / 1e6 / peaks["hbm_gbs"]}
    # roofline of the dominant kernel (in-place attention): algorithmic bytes per launch over its
    # mean launch time across both layers
    t_launch = float(np.mean([per[nm]["in_place_attn"]["ms"] for nm in per]))
    achieved = attn_bytes / t_launch / 1e6
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                "peak_source": "%s (copy bandwidth)" % peaks["source"],
                "kernel": "attn_fwd_kernel<%d, window>" % D}
    value = job_throughput(sum(flops), world, fused_ms_per_step)
    return {
        "metric": "shifted 3D window attention TFLOP/s (2 layers, attention in place on the grid)",
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": fused_ms_per_step, "higher_is_better": True,
        "packed_path": {"ms_per_step": ms_per_step,
                        "value": job_throughput(sum(flops), world, ms_per_step),
                        "note": "window pack -> varlen attention -> unpack per layer"},
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "tokens": n, "heads": H, "head_dim": D,
                   "l2": "inputs larger than L2 (%d MB per tensor)" % round(n * row / 1e6)},
        "layers": per, "roofline": roofline, "clocks": clocks,
        "gpu_launches": 2 * args.steps}


def run_vsa(args, rank, world, dev, h3, peaks):
    """Block-sparse video attention on the 1344x768 latent (32x48x84 grid, 4x4x4 blocks = 2016,
    top 252 = 1/8; 24 heads x 128): per step the block gate + top-k selection, then the attention
    of every query block over its selected blocks.  vsa_video_16x24x84 is a quarter of the grid
    for full ncu captures.  vsa_video_shared_half times the attention alone over a fixed synthetic
    selection in which paired query blocks share half of their 252 blocks (the gate is skipped)."""
    from workloads import vsa_paired_selection, vsa_video

    wl = vsa_video(grid=(16, 24, 84), topk=126) if args.workload == "vsa_video_16x24x84" else vsa_video()
    n, H, D = wl.num_tokens, wl.num_heads, wl.head_dim
    q, k, v = wl.q.to(dev), wl.k.to(dev), wl.v.to(dev)
    del wl.q, wl.k, wl.v
    nblk = h3.vsa_block_count(wl.grid, wl.block)
    scores = torch.empty((H, nblk, nblk), dtype=torch.float32, device=dev)
    sel = torch.empty((H, nblk, wl.topk), dtype=torch.int32, device=dev)
    ws = torch.empty(h3.vsa_select_workspace_size(wl.grid, wl.block, H, D), dtype=torch.uint8, device=dev)
    ws_attn = torch.empty(h3.vsa_attn_workspace_size(wl.grid, wl.block, H, wl.topk), dtype=torch.uint8,
                          device=dev)
    o = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    fixed_sel = args.workload == "vsa_video_shared_half"
    if fixed_sel:
        sel.copy_(torch.from_numpy(vsa_paired_selection(9, H, nblk, wl.topk, wl.topk // 2)))

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if not fixed_sel:
            h3.vsa_select(q, k, wl.grid, wl.topk, block=wl.block, scores=scores, out=sel, workspace=ws)
        if ev is not None:
            ev[1].record(stream)
        h3.vsa_attn_fwd(q, k, v, wl.grid, sel, block=wl.block, out=o, workspace=ws_attn)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if h3.get_device_error(dev) != 0:
        raise RuntimeError("device error during warm-up")
    # useful attention FLOPs from the selection: 4 H D sum_a n_a sum_{b in sel(a)} n_b
    sizes = torch.tensor(_block_sizes(wl.grid, wl.block), dtype=torch.float64, device=dev)
    flops = float(4.0 * D * (sizes[None, :, None] * sizes[sel.long()]).sum().item())
    # executed MMA work: query blocks 2p and 2p + 1 share a 128-row tile; a key block both of them
    # selected serves both halves of a step, so a pair sharing s of its topk blocks runs
    # ceil(s/2) + topk - s steps of a 128 x 128 QK^T and PV (the selection lists are distinct ids)
    sel_np = sel.cpu().numpy()
    first = sel_np[:, 0::2]
    second = sel_np[:, 1::2] if nblk % 2 == 0 else np.concatenate([sel_np[:, 1::2], first[:, -1:]], axis=1)
    member = np.zeros(second.shape[:2] + (nblk,), bool)
    np.put_along_axis(member, second.astype(np.int64), True, axis=2)
    shared = np.take_along_axis(member, first.astype(np.int64), axis=2).sum(axis=2)
    steps = (shared + 1) // 2 + wl.topk - shared
    flops_executed = float(steps.sum()) * 4.0 * 128 * 128 * D
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if h3.get_device_error(dev) != 0:
        raise RuntimeError("device error during the timed steps")
    ms_per_step = max_over_ranks(t0.elapsed_time(t1) / args.steps, world, dev)
    sel_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    attn_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    attn_tflops = flops / attn_ms / 1e9
    return {
        "metric": ("block-sparse video attention TFLOP/s (attention over a fixed selection: paired "
                   "query blocks share half their blocks)" if fixed_sel else
                   "block-sparse video attention TFLOP/s (gate + top-k + attention over selected blocks)"),
        "value": job_throughput(flops, world, ms_per_step), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "tokens": n, "heads": H, "head_dim": D, "blocks": nblk,
                   "topk": wl.topk, "attention_flop_useful": flops,
                   "l2": "inputs larger than L2 (%d MB per tensor)" % round(n * H * D * 2 / 1e6)},
        "kernels": {"select": {"ms": sel_ms, "note": "block means + fp32 score GEMM + radix top-k"},
                    "attn": {"ms": attn_ms, "tflops_useful": attn_tflops,
                             "tflops_executed": flops_executed / attn_ms / 1e9,
                             "shared_selection_frac": float(shared.mean() / wl.topk),
                             "steps": int(steps.sum()), "steps_unshared": int(steps.size * wl.topk),
                             "note": "each 128-row tile holds two query blocks; a step stacks two "
                                     "key blocks, and a block selected by only one of them is "
                                     "masked for the other half"}},
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": attn_tflops / peaks["bf16_tflops"], "traffic": None,
                     "kernel": "attn_fwd_kernel<%d, vsa>" % D,
                     "peak_source": peaks["source"] + " bf16_tflops (burst)",
                     "frac_of_sustained": attn_tflops / peaks["bf16_tflops_sustained"]},
        "clocks": clocks, "gpu_launches": (2 if fixed_sel else 5) * args.steps}


def run_continuation(args, rank, world, dev, h3, peaks):
    """Continuation window around the H3 request shape: the clip so far is one 5 s window (29
    latent frames of 40x50, 200 audio rows at 40 Hz), the next window has the same shape, rows are
    40 heads x 128 bf16 (10 KB).  Per step: pack the five row groups (+ positions, tags, target
    mask), one target-only row update over the packed sequence, append the new rows past the
    overlap to the clip."""
    H, D = 40, 128
    text, cf, ca, fh, fw, nf, na = 558, 29, 200, 40, 50, 29, 200
    cfg = h3.continuation_config(text, cf, ca, fh, fw, nf, na)
    plan = h3.continuation_plan(cfg)
    hw = fh * fw
    gen = torch.Generator(device=dev).manual_seed(8)
    mk = lambda n: torch.randn((n, H, D), generator=gen, device=dev).to(torch.bfloat16)
    t_rows, new_v, new_a = mk(text), mk(nf * hw), mk(na)
    clip_v = mk(plan.out_video_frames * hw)   # room for the append
    clip_a = mk(plan.out_audio_rows)
    n = plan.num_rows
    rows = torch.empty((n, H, D), dtype=torch.bfloat16, device=dev)
    upd = mk(n)
    row_bytes = H * D * 2
    stream = torch.cuda.current_stream(dev)
    # the clip's first cf frames / ca rows are its content; pack reads the tail from them
    src = dict(text=t_rows, clip_video=clip_v[:cf * hw], clip_audio=clip_a[:ca], new_video=new_v,
               new_audio=new_a)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        _, pos, tag, target = h3.continuation_pack(cfg, src["text"], src["clip_video"], src["clip_audio"],
                                                   src["new_video"], src["new_audio"], out=rows)
        if ev is not None:
            ev[1].record(stream)
        h3.masked_row_update(rows, upd, target)
        if ev is not None:
            ev[2].record(stream)
        h3.continuation_append(cfg, new_v, new_a, clip_v, clip_a)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if h3.get_device_error(dev) != 0:
        raise RuntimeError("device error during the timed steps")
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world, dev)
    n_tgt = n - plan.group_offset[3]
    pack_bytes = 2.0 * n * row_bytes + 14.0 * n              # rows in + out; pos 12 B, tag, target
    upd_bytes = 2.0 * n_tgt * row_bytes + n                   # target rows read + written; the mask
    app_rows = (nf - plan.keep_video_from) * hw + (na - plan.keep_audio_from)
    app_bytes = 2.0 * app_rows * row_bytes
    per = {}
    for name, a, b, nbytes in (("pack", 0, 1, pack_bytes), ("masked_update", 1, 2, upd_bytes),
                               ("append", 2, 3, app_bytes)):
        t = float(np.mean([e[a].elapsed_time(e[b]) for e in evs]))
        per[name] = {"ms": t, "bytes": nbytes, "gbs": nbytes / t / 1e6, "frac_hbm": nbytes / t / 1e6 / peaks["hbm_gbs"]}
    total_bytes = pack_bytes + upd_bytes + app_bytes
    achieved = per["pack"]["gbs"]
    return {
        "metric": "continuation window GB/s (pack + target-only update + append)",
        "value": world * total_bytes / ms / 1e6, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "continuation_h3_window_29x40x50_a200", "packed_rows": n,
                   "row_bytes": row_bytes, "start_frame": plan.start_frame, "audio_cut": plan.audio_cut,
                   "l2": "inputs larger than L2 (%.0f MB packed)" % (n * row_bytes / 1e6)},
        "kernels": per,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                     "kernel": "continuation_pack_kernel",
                     "peak_source": "%s (copy bandwidth)" % peaks["source"]},
        "clocks": clocks, "gpu_launches": 3 * args.steps}


def run_latency(args, rank, world, dev, h3):
    """The pages' worked example (45 tokens, segments [0,10,30,45], 2 x 64): launch-latency bound,
    so it is reported in microseconds per step (RoPE + attention plan + attention), issued
    eagerly and as one replayed CUDA graph."""
    import workloads

    wl = workloads.tiny_example(capacity=64)
    H, D, N = wl.num_heads, wl.head_dim, wl.num_tokens
    q, k, v = (t.to(dev) for t in (wl.q, wl.k, wl.v))
    pos, tag = torch.from_numpy(wl.pos).to(dev), torch.from_numpy(wl.tag).to(dev)
    cu, cu_req = torch.from_numpy(wl.cu_seqlens).to(dev), torch.from_numpy(wl.cu_requests).to(dev)
    frames = torch.from_numpy(wl.start_frames).to(dev)
    qr, kr, o = torch.empty_like(q), torch.empty_like(k), torch.empty_like(q)
    ws = torch.empty(max(16, h3.varlen_attn_workspace_size(wl.num_segments, H, wl.max_seqlen, D)),
                     dtype=torch.uint8, device=dev)

    def step():
        h3.rope_apply(q, k, pos, tag, cu_req, frames, num_tokens=N, q_out=qr, k_out=kr)
        h3.varlen_attn_fwd(qr, kr, v, cu, wl.max_seqlen, out=o, workspace=ws)

    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        for _ in range(max(3, args.warmup)):
            step()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    torch.cuda.synchronize(dev)
    if h3.get_device_error(dev) != 0:
        raise RuntimeError("device error during warm-up")
    reps = max(100, 100 * args.steps)

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for _ in range(reps):
                fn()
            e1.record(s)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / reps

    eager_us, graph_us = timed(step), timed(graph.replay)
    if h3.get_device_error(dev) != 0:
        raise RuntimeError("device error during the timed steps")
    return {
        "metric": "worked-example step latency (RoPE + varlen attention, 45 tokens)",
        "value": graph_us, "unit": "us", "n_gpus": world, "steps": reps, "warmup": max(3, args.warmup),
        "ms_per_step": graph_us / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "tokens": N, "cu_seqlens": [int(x) for x in wl.cu_seqlens],
                   "heads": H, "head_dim": D},
        "latency_us": {"cuda_graph_replay": graph_us, "eager": eager_us},
        "gpu_launches": 3 * reps}


def _block_sizes(grid, block):
    """Tokens per block (edge blocks cropped), in block-id order -- host bookkeeping for FLOPs."""
    axes = [np.array([min(b, L - b * i) for i in range((L + b - 1) // b)]) for L, b in zip(grid, block)]
    return np.einsum("i,j,k->ijk", *axes).reshape(-1)


def _kernel_sha():
    """Hash of the attention kernel's code with comments and whitespace removed: a comment edit
    keeps the DRAM traffic recorded for that code valid, any code change invalidates it."""
    import hashlib
    import re

    h = hashlib.sha256()
    for f in ("attn_fwd_sm103.cu", "sm103_ptx.cuh"):
        with open(os.path.join(ROOT, "packed_varlen_attention_modality_gb300", "csrc", f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(re.sub(r"\s+", " ", text).strip().encode())
    return h.hexdigest()[:16]


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
