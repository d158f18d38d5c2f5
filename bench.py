#!/usr/bin/env python
"""Benchmark of one position-split decode step (window + tail ring + LSE combine).

A step is one pass of the whole hot path over every layer of the workload: the
quantised-KV decode attention of the device window, the tail streamed from pinned
host memory through the prefetch ring, and the per-layer LSE combine.  The default
workload is the Qwen2.5-14B-like layer stack (48 layers, 40 q / 8 KV heads, head_dim
128, n_kv 65536, window 32768, fp16 K with 4 outlier channels per head, 3-slot ring).

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU oracle on a
bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn effective KV GB/s & % HBM peak; tail-hidden step ms vs max(compute,DMA)"
UNIT = "GB/s"


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="qwen14b_f16")
    ap.add_argument("--cpu-layers", type=int, default=0, help="layers in the oracle sample (0 = auto)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only this many layers (profiling of a small case; 0 = the workload's)")
    ap.add_argument("--auto-ring", action="store_true",
                    help="size the ring (slots, tile tokens) from the measured link and attention time "
                         "instead of the workload's fixed values")
    ap.add_argument("--v-fmt", default="",
                    help="with --kernel-only: store the window's V in this format instead "
                         "(f16, q8_0, tq2, tq3, tq4)")
    ap.add_argument("--k-fmt", default="",
                    help="with --kernel-only: store the window's K in this format instead "
                         "(f16, q8_0, or the V format's TurboQuant tier)")
    ap.add_argument("--ring-copy", choices=["engine", "kernel"], default="kernel",
                    help="how the ring moves tail tiles: the ring's copy kernel (default) or the copy engine")
    ap.add_argument("--n-q", type=int, default=1,
                    help="query tokens per step: > 1 runs verify-batch steps (batch 1, causal, the "
                         "query tokens at the cache's last positions)")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time the window decode-attention kernel alone on one layer of every "
                         "workload (one JSON line per workload; not the benchmark line)")
    return ap.parse_args(argv)


def max_over_ranks(torch, value: float, world: int, device) -> float:
    """The slowest rank's figure, on every rank (an all-reduce MAX over the job's process
    group; the identity for one rank)."""
    if world <= 1:
        return value
    tt = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    return float(tt.item())


def whole_job_rate(world: int, bytes_per_rank: float, ms_per_step: float) -> float:
    """Aggregate GB/s of the job: every rank (one replica of the workload) processes its
    own bytes each step, timed by the slowest rank."""
    return world * bytes_per_rank / (ms_per_step / 1e3) / 1e9


def step_distribution(per_step_ms):
    """Distribution of the timed steps' durations: median, 10th / 90th percentiles
    (linear interpolation between order statistics), extremes, and the number of
    steps longer than 1.25 x the median."""
    xs = sorted(float(x) for x in per_step_ms)
    if not xs:
        raise ValueError("no timed steps")

    def pct(p):
        pos = p * (len(xs) - 1)
        lo = int(pos)
        hi = min(lo + 1, len(xs) - 1)
        return xs[lo] + (xs[hi] - xs[lo]) * (pos - lo)

    p50 = statistics.median(xs)
    return {"p50_ms": p50, "p10_ms": pct(0.10), "p90_ms": pct(0.90), "min_ms": xs[0], "max_ms": xs[-1],
            "slow_steps": sum(1 for x in xs if x > 1.25 * p50)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# Arm CPU part numbers (the "CPU part" field of /proc/cpuinfo on Arm Linux hosts)
ARM_CPU_PARTS = {"0xd0c": "Arm Neoverse N1", "0xd40": "Arm Neoverse V1", "0xd49": "Arm Neoverse N2",
                 "0xd4f": "Arm Neoverse V2"}


def cpu_model(cpuinfo_text=None) -> str:
    """The host CPU's name: x86 "model name", or the Arm "CPU part" number (named when
    known)."""
    if cpuinfo_text is None:
        try:
            with open("/proc/cpuinfo") as f:
                cpuinfo_text = f.read()
        except OSError:
            return "unknown"
    for line in cpuinfo_text.splitlines():
        key = line.split(":", 1)[0].strip().lower()
        if key == "model name":
            return line.split(":", 1)[1].strip()
        if key == "cpu part":
            part = line.split(":", 1)[1].strip().lower()
            return f"{ARM_CPU_PARTS[part]} (CPU part {part})" if part in ARM_CPU_PARTS else f"CPU part {part}"
    return "unknown"


# ---------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------------
def _lib_signs(qps, synth, cfg):
    """The workload's TurboQuant sign words, or its Rotation, for the library."""
    w1, w2, block = synth.rotation_words(cfg)
    return w1 if w2 is None and block == 0 else qps.Rotation(w1, w2, block)


def time_oracle(cfg, n_layers: int):
    """Time the oracle's layer computation on ``n_layers`` layers of ``cfg`` (CPU).

    Returns (KV bytes processed, seconds, sample description).  The bytes are the
    stored KV planes of those layers, the same unit as the GPU figure."""
    import numpy as np

    import synth
    from oracle import pipeline

    from oracle import turboquant
    w1, w2, block = synth.rotation_words(cfg)
    signs = w1.numpy() if w2 is None and block == 0 else turboquant.Rotation(
        w1.numpy(), None if w2 is None else w2.numpy(), block or None)
    nbytes = 0
    elapsed = 0.0
    for layer in range(n_layers):
        q = synth.query_f16(cfg, layer).numpy()
        k = synth.kv_f16(cfg, layer, "k", cfg.n_kv).numpy()
        v = synth.kv_f16(cfg, layer, "v", cfg.n_kv).numpy()
        t0 = time.perf_counter()
        pipeline.mixed_layer_reference(q, k, v, cfg.wc, cfg.k_fmt, cfg.v_fmt, cfg.tk_fmt, cfg.tv_fmt,
                                       cfg.scale, cfg.softcap, signs)
        elapsed += time.perf_counter() - t0
        for fmt, x in ((cfg.k_fmt, k[:cfg.wc]), (cfg.v_fmt, v[:cfg.wc]), (cfg.tk_fmt, k[cfg.wc:]),
                       (cfg.tv_fmt, v[cfg.wc:])):
            if x.shape[0]:
                nbytes += sum(p.nbytes for p in pipeline.encode(fmt, x[:1], signs)) * x.shape[0]
        del q, k, v
    sample = (f"{n_layers} of {cfg.layers} layers of {cfg.name}, all {cfg.hq} query heads over all "
              f"{cfg.n_kv} positions (window + tail), float64")
    return nbytes, elapsed, sample


def oracle_layers_for(cfg, requested: int) -> int:
    if requested > 0:
        return min(requested, cfg.layers)
    return min(cfg.layers, 4 if cfg.d <= 128 else 1)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import synth

    cfg = synth.by_name(args.config)
    steps = max(1, args.steps)
    layers = oracle_layers_for(cfg, args.cpu_layers)
    for _ in range(max(0, min(args.warmup, 1))):
        time_oracle(cfg, 1)
    total_b, total_s = 0, 0.0
    sample = ""
    for _ in range(steps):
        b, s, sample = time_oracle(cfg, layers)
        total_b += b
        total_s += s
    value = total_b / total_s / 1e9
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": 1000.0 * total_s / steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1), outlier K channels)",
        "config": {"workload": cfg.name, "layers": cfg.layers, "hq": cfg.hq, "hkv": cfg.hkv, "d": cfg.d,
                   "n_kv": cfg.n_kv, "wc": cfg.wc, "k_fmt": cfg.k_fmt, "v_fmt": cfg.v_fmt},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                         "sample": sample + f", per step; CPU {cpu_model()}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    return 0


# ---------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.path = tempfile.mktemp(prefix="qps_clocks_", suffix=".csv")
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------
# measured peaks and committed ncu traffic
# ---------------------------------------------------------------------------------
def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def attention_source_sha():
    csrc = os.path.join(ROOT, "quantized_position_split_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.startswith("attn") or name.endswith((".h", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def window_signature(cfg):
    """What decides the window launch's kernel and its bytes: shapes, window length,
    formats, softcap and rotation (not the layer count or the tail's formats)."""
    return (cfg.kind, cfg.batch, cfg.hq, cfg.hkv, cfg.d, cfg.wc, cfg.k_fmt, cfg.v_fmt, cfg.softcap,
            cfg.sign_seed, cfg.sign_seed2, cfg.rot_block)


def traffic_workload(cfg, configs) -> str:
    """The workload whose window-kernel DRAM traffic file serves ``cfg``: ``cfg`` itself,
    or the workload whose window launch is the same kernel on the same window (a
    mixed-format tail changes only the tail's kernels)."""
    if not cfg.mixed:
        return cfg.name
    for c in configs:
        if not c.mixed and window_signature(c) == window_signature(cfg):
            return c.name
    return cfg.name


def committed_traffic(workload: str):
    path = os.path.join(ROOT, "profiles", f"attn_window_{workload}_traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)
    except (OSError, ValueError):
        return None
    if j.get("kernel_source_sha") != attention_source_sha():
        return None  # counters were taken on another version of the kernel
    return j.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------------
def measure_link(torch, device, nbytes=1 << 30):
    """Pinned host -> device copy bandwidth (one 1 GiB cudaMemcpyAsync, best of 4), and
    a single-thread host memcpy of the same size."""
    import numpy as np

    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s = torch.cuda.current_stream()
    best = 0.0
    for _ in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        dst.copy_(src, non_blocking=True)
        e1.record(s)
        e1.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    a = np.ones(nbytes // 4, dtype=np.float32)
    b = np.empty_like(a)
    t0 = time.perf_counter()
    np.copyto(b, a)
    host = a.nbytes / (time.perf_counter() - t0) / 1e9
    del src, dst, a, b
    return best, host


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())

    import synth
    import quantized_position_split_gb300 as qps
    from quantized_position_split_gb300 import build as qbuild
    from quantized_position_split_gb300.decode import PositionSplitDecoder

    qbuild.build()
    cfg = synth.by_name(args.config)
    if args.layers > 0:
        cfg = cfg.replace(layers=min(args.layers, cfg.layers))
    if cfg.kind != "split":
        raise SystemExit("bench.py times the position-split workloads")
    signs = _lib_signs(qps, synth, cfg)
    ring_plan = None
    if args.auto_ring:
        from quantized_position_split_gb300 import autosize
        link, host = autosize.measure_link(device)
        bw_eff = link  # pinned host -> device through the copy engine: the tail's own path
        att_ms = autosize.attention_ms(cfg.k_fmt, cfg.v_fmt, batch=cfg.batch, hq=cfg.hq, hkv=cfg.hkv, d=cfg.d,
                                       n_kv=cfg.n_kv, scale=cfg.scale, softcap=cfg.softcap, signs=signs,
                                       device=device)
        ptb = cfg.hkv * (sum(qps.plane_row_bytes(cfg.tk_fmt, cfg.d)) + sum(qps.plane_row_bytes(cfg.tv_fmt, cfg.d)))
        slot_budget = 4.0 * (1 << 30)  # device memory set aside for the ring's slots
        rp = qps.plan_ring(att_ms, bw_eff, slot_budget, float(cfg.tail_len * ptb))
        tile_tokens = max(16, int(rp["tile_bytes"] // ptb) // 16 * 16)
        ring_plan = dict(rp, link_gbs=link, host_memcpy_gbs=host, bw_eff_gbs=bw_eff, attention_ms=att_ms,
                         slot_budget_bytes=slot_budget, tile_tokens=tile_tokens)
        cfg = cfg.replace(ring_slots=rp["n_slots"], tile_tokens=tile_tokens)
    dec = PositionSplitDecoder(layers=cfg.layers, batch=cfg.batch, hq=cfg.hq, hkv=cfg.hkv, d=cfg.d,
                               n_kv=cfg.n_kv, wc=cfg.wc, k_fmt=cfg.k_fmt, v_fmt=cfg.v_fmt,
                               scale=cfg.scale, softcap=cfg.softcap, signs=signs,
                               ring_slots=cfg.ring_slots, tile_tokens=cfg.tile_tokens, device=device,
                               tail_k_fmt=cfg.tail_k_fmt, tail_v_fmt=cfg.tail_v_fmt, ring_copy=args.ring_copy,
                               n_q=args.n_q)
    for layer in range(cfg.layers):
        q = (synth.query_f16(cfg, layer, device=device) if args.n_q == 1 else
             synth.randn_f16((1, args.n_q, cfg.hq, cfg.d), cfg.seed, cfg.name, "verify", layer, device=device))
        k = synth.kv_f16(cfg, layer, "k", cfg.n_kv, device=device)
        v = synth.kv_f16(cfg, layer, "v", cfg.n_kv, device=device)
        dec.load_layer(layer, k, v, q)
        del q, k, v
    dec.build()
    torch.cuda.synchronize()

    link_gbs, host_memcpy_gbs = measure_link(torch, device)
    stream = torch.cuda.current_stream()
    window_bytes = dec.window_bytes()
    tail_bytes = dec.tail_bytes()
    kv_bytes = window_bytes + tail_bytes

    # per-layer timing events around the window part, one pair per (step, layer)
    K, W, L = args.steps, args.warmup, cfg.layers
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
          for _ in range(K)]
    for row in ev:
        for a, b in row:
            a.record(stream)
            b.record(stream)

    def set_events(step_events):
        for layer in range(L):
            pe = dec.plan.layers[layer].part_events
            if step_events is None:
                pe[0] = pe[1] = None
            else:
                pe[0], pe[1] = step_events[layer][0].cuda_event, step_events[layer][1].cuda_event

    set_events(None)
    for _ in range(W):
        dec.step(stream)
    # window-only steps (ring and tail omitted) for the step criterion
    for _ in range(2):
        dec.window_step(stream)
    torch.cuda.synchronize()
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(K):
        dec.window_step(stream)
    w1.record(stream)
    torch.cuda.synchronize()
    window_step_ms = w0.elapsed_time(w1) / K

    # the timed region
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        gpu_id = None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_id)
    time.sleep(0.3)
    qps.launch_count(reset=True)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    bounds = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.nvtx.range_push("qps_timed")  # lets a profiler select the timed launches
    t0.record(stream)
    for i in range(K):
        set_events(ev[i])
        dec.step(stream)
        bounds[i].record(stream)
    t1.record(stream)
    torch.cuda.nvtx.range_pop()
    launches = qps.launch_count()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    set_events(None)
    step_ms = max_over_ranks(torch, t0.elapsed_time(t1) / K, world, device)
    win_ms = [ev[i][layer][0].elapsed_time(ev[i][layer][1]) for i in range(K) for layer in range(L)]
    win_launch_ms = statistics.mean(win_ms)
    per_step = [t0.elapsed_time(bounds[0])] + [bounds[i - 1].elapsed_time(bounds[i]) for i in range(1, K)]
    step_dist = step_distribution(per_step)

    # end to end through the public API with host buffers: q in, (o, lse) out each step
    q_host = torch.empty_like(dec.q, device="cpu").pin_memory()
    q_host.copy_(dec.q.cpu())
    o_host = torch.empty_like(dec.o, device="cpu").pin_memory()
    lse_host = torch.empty_like(dec.lse, device="cpu").pin_memory()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        dec.q.copy_(q_host, non_blocking=True)
        dec.step(stream)
        o_host.copy_(dec.o, non_blocking=True)
        lse_host.copy_(dec.lse, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / K
    h2d = q_host.numel() * q_host.element_size()
    d2h = o_host.numel() * o_host.element_size() + lse_host.numel() * lse_host.element_size()
    e2e_ms = max_over_ranks(torch, e2e_ms, world, device)

    dec.ring.sync()

    # roofline of the dominant kernel: the window decode-attention launch
    per_launch_bytes = window_bytes / L
    rows = dec.rows
    n_split_w = qps.attn_plan(dec.window_args[0])[0]
    q_bytes = rows * cfg.d * 2
    part_bytes = n_split_w * rows * (cfg.d + 1) * 4
    algo_bytes = per_launch_bytes + q_bytes + part_bytes
    peak, peak_kind = measured_hbm_peak()
    achieved = algo_bytes / (win_launch_ms / 1e3) / 1e9
    tail_dma_ms = tail_bytes / (link_gbs * 1e9) * 1e3
    bound_ms = max(window_step_ms, tail_dma_ms)

    if rank != 0:
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        b, s, sample = time_oracle(cfg, oracle_layers_for(cfg, args.cpu_layers))
        cpu = {"value": b / s / 1e9, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": sample + f"; CPU {cpu_model()}"}
    value = whole_job_rate(world, kv_bytes, step_ms)
    out = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("f16" if cfg.k_fmt == "f16" and cfg.v_fmt == "f16" else f"{cfg.k_fmt}/{cfg.v_fmt}") +
                 (f" window, {cfg.tk_fmt}/{cfg.tv_fmt} tail" if cfg.mixed else ""),
        "data": "synthetic (seeded N(0,1) fp16, 4 outlier K channels per head x20)",
        "config": {"workload": cfg.name, "layers": cfg.layers, "batch": cfg.batch, "hq": cfg.hq,
                   "hkv": cfg.hkv, "d": cfg.d, "n_kv": cfg.n_kv, "wc": cfg.wc, "k_fmt": cfg.k_fmt,
                   "v_fmt": cfg.v_fmt, "tail_k_fmt": cfg.tk_fmt, "tail_v_fmt": cfg.tv_fmt,
                   "softcap": cfg.softcap, "ring_slots": cfg.ring_slots,
                   "tile_tokens": cfg.tile_tokens, "ring_plan": ring_plan, "ring_copy": args.ring_copy, "n_q": args.n_q,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (window %.2f GB + tail %.2f GB per step)" %
                         (window_bytes / 1e9, tail_bytes / 1e9)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": committed_traffic(traffic_workload(cfg, synth.CONFIGS)),
                     "kernel": "window decode attention (one launch per layer)",
                     "algorithmic_bytes_per_launch": algo_bytes, "launch_ms": win_launch_ms,
                     "peak_source": peak_kind},
        # the ring's tail transfer: most of the step's GPU time goes to the ring copy
        # kernel (or the copy engine), bound by the host link rather than by HBM
        "roofline_tail": {"bound": "host link", "achieved": tail_bytes / (step_ms / 1e3) / 1e9,
                          "peak": link_gbs, "unit": "GB/s",
                          "frac": tail_bytes / (step_ms / 1e3) / 1e9 / link_gbs,
                          "kernel": ("ring copy kernel" if args.ring_copy == "kernel" else "copy engine") +
                                    " (tail tiles, pinned host -> ring slot)",
                          "achieved_source": "tail bytes per step / step time",
                          "peak_source": "pinned 1 GiB host-to-device cudaMemcpyAsync, best of 4, this run"},
        "step": {"ms": step_ms, "window_only_ms": window_step_ms, "tail_dma_ms": tail_dma_ms,
                 "bound_ms": bound_ms, "ratio_to_bound": step_ms / bound_ms,
                 "tail_stream_gbs": tail_bytes / (step_ms / 1e3) / 1e9,
                 "link_probe_gbs": link_gbs, "host_memcpy_1thread_gbs": host_memcpy_gbs,
                 "steps_per_s": 1000.0 / step_ms, "per_step": step_dist},
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_rate(world, kv_bytes, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "clocks": clk,
    }
    print(json.dumps(out), flush=True)
    dec.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# kernel-only lines of a workload's window with (K, V) stored in other formats: V at the
# other TurboQuant tiers, and K and V both TurboQuant (K read in the rotated domain)
TIER_VARIANTS = {"qwen14b_q8": (("q8_0", "tq4"), ("q8_0", "tq2"), ("tq4", "tq4"), ("tq3", "tq3"), ("tq2", "tq2")),
                 "gemma_global_q8k_tq3v": (("q8_0", "tq4"), ("q8_0", "tq2"), ("tq3", "tq3"))}


def run_kernel_only(args):
    """Per-launch time of the window decode-attention kernel on one layer of each
    workload (or of --config), timed back to back with CUDA events; inputs > L2 except
    the tiny and fan-out workloads (flagged)."""
    import torch

    import synth
    import quantized_position_split_gb300 as qps
    from quantized_position_split_gb300 import build as qbuild

    qbuild.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    # (the mixed-tail workloads share their window kernel with the uniform ones)
    names = [args.config] if args.config != "qwen14b_f16" or args.layers else [
        c.name for c in synth.CONFIGS if not c.mixed]
    peak, peak_kind = measured_hbm_peak()
    s = torch.cuda.current_stream()
    for name in names:
        cfg = synth.by_name(name)
        if args.v_fmt or args.k_fmt:
            cfg = cfg.replace(v_fmt=args.v_fmt or cfg.v_fmt, k_fmt=args.k_fmt or cfg.k_fmt)
            name = f"{name} K={cfg.k_fmt} V={cfg.v_fmt}"
        signs = _lib_signs(qps, synth, cfg)
        if cfg.kind == "split":
            q = synth.query_f16(cfg, 0, device=dev)
            k = synth.kv_f16(cfg, 0, "k", cfg.wc, device=dev)
            v = synth.kv_f16(cfg, 0, "v", cfg.wc, device=dev)
            K = qps.encode_kv_head_major(cfg.k_fmt, k, signs)
            V = qps.encode_kv_head_major(cfg.v_fmt, v, signs)
            a = qps.attn_args(q, K, V, scale=cfg.scale, softcap=cfg.softcap, v_signs=signs)
            rows = cfg.batch * cfg.hq
        else:
            q = synth.randn_f16((cfg.agents, cfg.hq, cfg.d), cfg.seed, cfg.name, "q", device=dev)
            pk = synth.randn_f16((cfg.n_kv, cfg.hkv, cfg.d), cfg.seed, cfg.name, "prefix", "k", device=dev)
            pv = synth.randn_f16((cfg.n_kv, cfg.hkv, cfg.d), cfg.seed, cfg.name, "prefix", "v", device=dev)
            K = qps.encode_kv_head_major(cfg.k_fmt, pk, signs)
            V = qps.encode_kv_head_major(cfg.v_fmt, pv, signs)
            a = qps.attn_args(q, K, V, scale=cfg.scale, softcap=cfg.softcap, v_signs=signs, shared=True)
            rows = cfg.agents * cfg.hq
        for n_q in ([1, 4] if name == "qwen14b_q8" and cfg.kind == "split" else [1]):
            if n_q > 1:  # a verify batch: 4 query tokens at the end of the window, causal
                q4 = synth.randn_f16((cfg.batch, n_q, cfg.hq, cfg.d), cfg.seed, cfg.name, "verify", device=dev)
                a = qps.attn_args(q4, K, V, scale=cfg.scale, softcap=cfg.softcap, v_signs=signs,
                                  q_pos=cfg.wc - n_q)
                rows = cfg.batch * n_q * cfg.hq
            _time_window_launch(qps, torch, a, name if n_q == 1 else f"{name} verify n_q={n_q} causal",
                                rows, cfg, K, V, dev, s, peak, peak_kind)
        # the same window with (K, V) in the other formats
        for kf, vf in (TIER_VARIANTS.get(name, ()) if not (args.layers or args.v_fmt or args.k_fmt) else ()):
            del K, V
            K = qps.encode_kv_head_major(kf, k, signs)
            V = qps.encode_kv_head_major(vf, v, signs)
            a = qps.attn_args(q, K, V, scale=cfg.scale, softcap=cfg.softcap, v_signs=signs)
            _time_window_launch(qps, torch, a, f"{name} K={kf} V={vf}", cfg.batch * cfg.hq,
                                cfg.replace(k_fmt=kf, v_fmt=vf), K, V, dev, s, peak, peak_kind)
        qps.device_status(reset=True)
    return 0


def _time_window_launch(qps, torch, a, label, rows, cfg, K, V, dev, s, peak, peak_kind):
    """Per-launch time of one window attention (50 launches back to back, CUDA events)."""
    n_split, _ = qps.attn_plan(a)
    parts = (torch.empty((n_split, rows, cfg.d), device=dev), torch.empty((n_split, rows), device=dev))
    for _ in range(3):
        qps.attn_decode_window(a, parts=parts)
    n = 50
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(s)
    for _ in range(n):
        qps.attn_decode_window(a, parts=parts)
    e1.record(s)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / n * 1e3
    kv = K.nbytes() + V.nbytes()
    algo = kv + rows * cfg.d * 2 + n_split * rows * (cfg.d + 1) * 4
    print(json.dumps({"kernel": "attn_decode_window", "workload": label, "path": qps.attn_path(a),
                      "n_split": n_split, "launch_us": us, "kv_bytes": kv, "algorithmic_bytes": algo,
                      "achieved_gbs": algo / us / 1e3, "frac_of_hbm": algo / us / 1e3 / peak,
                      "peak_gbs": peak, "peak_source": peak_kind,
                      "l2_resident": kv < 129e6}), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel_only:
        return run_kernel_only(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
