#!/usr/bin/env python
"""Benchmark of one position-split decode step (window + tail ring + LSE combine).

A step is one pass of the whole hot path over every layer of the workload: the
quantised-KV decode attention of the device window, the tail streamed from pinned
host memory through the prefetch ring, and the per-layer LSE combine.  The default
workload is the largest single-GPU configuration, the Qwen2.5-14B-like layer stack
with K and V at q8_0 (48 layers, 40 q / 8 KV heads, head_dim 128, n_kv 131072, window
98304 on the device, a 32768-position compressed tail streamed through a 3-slot ring).

The same JSON line carries one sub-record per other workload (``--sub-configs``): the
fp16 Qwen-like stack, the Gemma-like global layers (q8_0 K / 3-bit TurboQuant V,
head_dim 512, softcap 50) and the shared-prefix fan-out.  Every record is checked: the
device error word of the bounded in-kernel waits after the timed and the end-to-end
steps (a wait that gave up exits non-zero), and the outputs of sampled layers against
the float64 CPU oracle on the same inputs, whose timing is the ``cpu_baseline``.

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU oracle on a
bounded sample of the same workload instead.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attn effective KV GB/s & % HBM peak; tail-hidden step ms vs max(compute,DMA)"
UNIT = "GB/s"
DEFAULT_CONFIG = "qwen14b_q8"
SUB_CONFIGS = "qwen14b_f16,gemma_global_q8k_tq3v,fanout_prefix"
# the bar every output is held to: per query row rel-L2 and max-abs of O, |dLSE|
PARITY_BAR = {"rel_l2": 1e-3, "max_abs": 2e-3, "dlse": 1e-4}
L2_BYTES = 129e6
DATA = "synthetic (seeded N(0,1) fp16, 4 outlier K channels per head x20)"


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--sub-configs", default=SUB_CONFIGS,
                    help="comma-separated workloads measured as sub-records of the same line ('' for none)")
    ap.add_argument("--cpu-layers", type=int, default=0, help="layers in the oracle sample (0 = auto)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only this many layers (profiling of a small case; 0 = the workload's)")
    ap.add_argument("--auto-ring", action="store_true",
                    help="size the ring (slots, tile tokens) from the measured link and attention time "
                         "instead of the workload's fixed values")
    ap.add_argument("--tile-tokens", type=int, default=0,
                    help="positions per ring tile of the line's workload (0 = the workload's; "
                         "--auto-ring sizes it instead)")
    ap.add_argument("--n-split-window", type=int, default=0,
                    help="split count of the window launches (0 = the library's automatic choice)")
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
# workload description shared by both arms
# ---------------------------------------------------------------------------------
# bytes per stored row of each plane of a format (data, aux, aux2), head_dim d
ROW_BYTES = {"f16": lambda d: [2 * d], "q8_0": lambda d: [d, d // 16], "tq3": lambda d: [d // 4, d // 8, 2],
             "tq2": lambda d: [d // 4, 2], "tq4": lambda d: [d // 2, 2]}


def _pad16(n: int) -> int:
    return (n + 15) // 16 * 16


def split_kv_bytes(cfg):
    """(window, tail) bytes one step reads: every stored plane of every layer, each KV
    head's positions padded to 16 rows as the decoder stores them (head-major)."""
    row = lambda fk, fv: sum(ROW_BYTES[fk](cfg.d)) + sum(ROW_BYTES[fv](cfg.d))  # noqa: E731
    window = cfg.layers * cfg.hkv * _pad16(cfg.wc) * row(cfg.k_fmt, cfg.v_fmt) if cfg.wc > 0 else 0
    tail = 0
    for a in range(0, cfg.tail_len, cfg.tile_tokens):
        n = min(cfg.tile_tokens, cfg.tail_len - a)
        tail += cfg.hkv * _pad16(n) * row(cfg.tk_fmt, cfg.tv_fmt)
    return window, tail * cfg.layers


# host time the reference arm's oracle sample may take over a whole run (seconds)
REFERENCE_BUDGET_S = 150.0


def line_workload(synth, args):
    """The workload the line times, as both arms build it: ``--config`` cut to
    ``--layers`` and with ``--tile-tokens`` positions per ring tile."""
    cfg = synth.by_name(args.config)
    if args.layers > 0:
        cfg = cfg.replace(layers=min(args.layers, cfg.layers))
    if args.tile_tokens > 0:
        cfg = cfg.replace(tile_tokens=args.tile_tokens)
    return cfg


def bench_config(cfg, args, ring_plan=None) -> dict:
    """The line's ``config``: the workload and the launch configuration timed (the same
    dict on both arms for the same arguments)."""
    if cfg.kind == "fanout":
        pre = cfg.hkv * _pad16(cfg.n_kv) * (sum(ROW_BYTES[cfg.k_fmt](cfg.d)) + sum(ROW_BYTES[cfg.v_fmt](cfg.d)))
        suf = cfg.agents * cfg.hkv * _pad16(cfg.suffix_len) * 2 * 2 * cfg.d
        return {"workload": cfg.name, "layers": cfg.layers, "agents": cfg.agents, "hq": cfg.hq, "hkv": cfg.hkv,
                "d": cfg.d, "prefix_len": cfg.n_kv, "suffix_len": cfg.suffix_len, "k_fmt": cfg.k_fmt,
                "v_fmt": cfg.v_fmt, "suffix_fmt": "f16", "softcap": cfg.softcap,
                "parallelism": f"replicas x{args.gpus}",
                "l2": "inputs smaller than L2 (prefix %.2f MB + suffixes %.2f MB): L2 flushed (256 MB "
                      "write) before every timed step" % (pre / 1e6, suf / 1e6)}
    window, tail = split_kv_bytes(cfg)
    return {"workload": cfg.name, "layers": cfg.layers, "batch": cfg.batch, "hq": cfg.hq,
            "hkv": cfg.hkv, "d": cfg.d, "n_kv": cfg.n_kv, "wc": cfg.wc, "k_fmt": cfg.k_fmt,
            "v_fmt": cfg.v_fmt, "tail_k_fmt": cfg.tk_fmt, "tail_v_fmt": cfg.tv_fmt,
            "softcap": cfg.softcap, "ring_slots": cfg.ring_slots,
            "tile_tokens": cfg.tile_tokens, "ring_plan": ring_plan, "ring_copy": args.ring_copy, "n_q": args.n_q,
            "n_split_window": args.n_split_window or "auto",
            "parallelism": f"replicas x{args.gpus}",
            "l2": "inputs larger than L2 (window %.2f GB + tail %.2f GB per step)" % (window / 1e9, tail / 1e9)}


# ---------------------------------------------------------------------------------
# CPU oracle: timing (the reference arm and the cpu_baseline leg) and the check of the
# GPU outputs
# ---------------------------------------------------------------------------------
def _lib_signs(qps, synth, cfg):
    """The workload's TurboQuant sign words, or its Rotation, for the library."""
    w1, w2, block = synth.rotation_words(cfg)
    return w1 if w2 is None and block == 0 else qps.Rotation(w1, w2, block)


def _oracle_signs(synth, cfg):
    from oracle import turboquant
    w1, w2, block = synth.rotation_words(cfg)
    return w1.numpy() if w2 is None and block == 0 else turboquant.Rotation(
        w1.numpy(), None if w2 is None else w2.numpy(), block or None)


def parity_figures(o_gpu, lse_gpu, o_ref, lse_ref) -> dict:
    """Worst per-row rel-L2 and max-abs of O and |dLSE| of one layer (float64); rows
    empty on one side only count as a failure."""
    import numpy as np

    o_gpu = np.asarray(o_gpu, dtype=np.float64).reshape(o_ref.shape)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64).reshape(lse_ref.shape)
    diff = o_gpu - o_ref
    den = np.linalg.norm(o_ref, axis=-1)
    rel = np.linalg.norm(diff, axis=-1) / np.where(den > 0, den, 1.0)
    fin = np.isfinite(lse_ref)
    dl = np.abs(lse_gpu[fin] - lse_ref[fin])
    bad = not np.array_equal(fin, np.isfinite(lse_gpu))
    return {"rel_l2": float(rel.max()), "max_abs": float(np.abs(diff).max()),
            "dlse": float("inf") if bad else (float(dl.max()) if dl.size else 0.0)}


def merge_parity(figs) -> dict:
    out = {k: max(f[k] for f in figs) for k in PARITY_BAR}
    out["pass"] = all(out[k] <= PARITY_BAR[k] for k in PARITY_BAR)
    out["bar"] = dict(PARITY_BAR)
    return out


def time_oracle(cfg, layers, device="cpu", gpu_outputs=None):
    """Time the oracle's layer computation on the given ``layers`` of ``cfg`` (CPU).

    Inputs are drawn from the seeded generators on ``device`` (the device the GPU path
    drew them on, so that they are the same values) and copied to host before the
    clock starts.  ``gpu_outputs(layer)`` -> (O, lse) host arrays of the GPU path:
    when given, each oracle layer is compared with it.  Returns (KV bytes processed,
    seconds, sample description, parity figures or None).  The bytes are the stored
    KV planes of those layers, the same unit as the GPU figure."""
    import synth
    from oracle import pipeline

    signs = _oracle_signs(synth, cfg)
    nbytes = 0
    elapsed = 0.0
    figs = []
    for layer in layers:
        q = synth.query_f16(cfg, layer, device=device).cpu().numpy()
        k = synth.kv_f16(cfg, layer, "k", cfg.n_kv, device=device).cpu().numpy()
        v = synth.kv_f16(cfg, layer, "v", cfg.n_kv, device=device).cpu().numpy()
        t0 = time.perf_counter()
        ro, rl = pipeline.mixed_layer_reference(q, k, v, cfg.wc, cfg.k_fmt, cfg.v_fmt, cfg.tk_fmt, cfg.tv_fmt,
                                                cfg.scale, cfg.softcap, signs)
        elapsed += time.perf_counter() - t0
        for fmt, x in ((cfg.k_fmt, k[:cfg.wc]), (cfg.v_fmt, v[:cfg.wc]), (cfg.tk_fmt, k[cfg.wc:]),
                       (cfg.tv_fmt, v[cfg.wc:])):
            if x.shape[0]:
                nbytes += sum(p.nbytes for p in pipeline.encode(fmt, x[:1], signs)) * x.shape[0]
        if gpu_outputs is not None:
            o, lse = gpu_outputs(layer)
            figs.append(parity_figures(o, lse, ro.reshape(-1, cfg.d), rl.reshape(-1)))
        del q, k, v
    sample = (f"layers {list(layers)} of {cfg.layers} of {cfg.name}, all {cfg.hq} query heads over all "
              f"{cfg.n_kv} positions (window + tail), float64")
    par = None
    if figs:
        par = merge_parity(figs)
        par["layers"] = list(layers)
    return nbytes, elapsed, sample, par


def oracle_layers_for(cfg, requested: int):
    """The oracle sample: the first and the last layer plus evenly spaced ones between
    (4 layers at head_dim <= 128, 1 at 512, or ``requested``)."""
    n = min(requested, cfg.layers) if requested > 0 else min(cfg.layers, 4 if cfg.d <= 128 else 1)
    if n <= 1:
        return [cfg.layers - 1]
    return sorted({round(i * (cfg.layers - 1) / (n - 1)) for i in range(n)})


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import synth

    cfg = line_workload(synth, args)
    if cfg.kind != "split":
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the position-split "
                          "workloads only"}), flush=True)
        return 0
    steps = max(1, args.steps)
    layers = oracle_layers_for(cfg, args.cpu_layers)
    # one untimed layer warms up and gives the wall time of a layer (inputs included);
    # each step then takes as many of the sample layers, in turn, as keep the whole run
    # near REFERENCE_BUDGET_S of host time
    t_w = time.perf_counter()
    time_oracle(cfg, layers[:1])
    per_layer = max(time.perf_counter() - t_w, 1e-3)
    per_step = max(1, min(len(layers), int(REFERENCE_BUDGET_S / steps / per_layer)))
    total_b, total_s = 0, 0.0
    sample = ""
    for i in range(steps):
        pick = [layers[(i * per_step + j) % len(layers)] for j in range(per_step)]
        b, s, sample, _ = time_oracle(cfg, pick)
        total_b += b
        total_s += s
    if per_step < len(layers):
        sample += f" (each step {per_step} of the layers {layers} in turn)"
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
        "data": DATA,
        "config": bench_config(cfg, args),
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


def attention_source_sha(root=None):
    csrc = os.path.join(root or ROOT, "quantized_position_split_gb300", "csrc")
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


def committed_traffic(workload: str, root=None):
    """DRAM bytes per window launch from the committed ncu capture of ``workload``, or
    None when there is none or it was taken on another version of the kernels."""
    root = root or ROOT
    path = os.path.join(root, "profiles", f"attn_window_{workload}_traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)
    except (OSError, ValueError):
        return None
    if j.get("kernel_source_sha") != attention_source_sha(root):
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


class DeviceCheckFailed(RuntimeError):
    pass


def check_device(qps, where: str):
    """Raise if a kernel's bounded wait gave up since the last reset: the outputs of
    the steps just timed are invalid, and so is any figure taken from them."""
    from quantized_position_split_gb300 import _native as N
    try:
        qps.device_status(reset=False)
    except N.QpsError as e:
        raise DeviceCheckFailed(f"device status after {where}: {e}") from e


def build_split(torch, qps, synth, cfg, args, device, n_q=1):
    """A PositionSplitDecoder with every layer of ``cfg`` loaded from the seeded
    generators on ``device`` (the oracle check draws the same values there)."""
    from quantized_position_split_gb300.decode import PositionSplitDecoder

    dec = PositionSplitDecoder(layers=cfg.layers, batch=cfg.batch, hq=cfg.hq, hkv=cfg.hkv, d=cfg.d,
                               n_kv=cfg.n_kv, wc=cfg.wc, k_fmt=cfg.k_fmt, v_fmt=cfg.v_fmt,
                               scale=cfg.scale, softcap=cfg.softcap, signs=_lib_signs(qps, synth, cfg),
                               ring_slots=cfg.ring_slots, tile_tokens=cfg.tile_tokens, device=device,
                               tail_k_fmt=cfg.tail_k_fmt, tail_v_fmt=cfg.tail_v_fmt, ring_copy=args.ring_copy,
                               n_q=n_q, n_split_window=args.n_split_window)
    for layer in range(cfg.layers):
        q = (synth.query_f16(cfg, layer, device=device) if n_q == 1 else
             synth.randn_f16((1, n_q, cfg.hq, cfg.d), cfg.seed, cfg.name, "verify", layer, device=device))
        k = synth.kv_f16(cfg, layer, "k", cfg.n_kv, device=device)
        v = synth.kv_f16(cfg, layer, "v", cfg.n_kv, device=device)
        dec.load_layer(layer, k, v, q)
        del q, k, v
    dec.build()
    torch.cuda.synchronize()
    return dec


def time_split_steps(torch, qps, dec, K, W, stream, world, device, gpu_id):
    """Warm-up, the window-only steps, the timed steps (per-layer events around the
    window part, clocks sampled) and the end-to-end steps through host buffers; the
    device error word is checked after each."""
    L = dec.layers
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
    check_device(qps, "the warm-up and window-only steps")

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
    check_device(qps, "the timed steps")
    step_ms = max_over_ranks(torch, t0.elapsed_time(t1) / K, world, device)
    win_ms = [ev[i][layer][0].elapsed_time(ev[i][layer][1]) for i in range(K) for layer in range(L)]
    per_step = [t0.elapsed_time(bounds[0])] + [bounds[i - 1].elapsed_time(bounds[i]) for i in range(1, K)]

    # end to end through the public API with host buffers: q in, (o, lse) out each step,
    # moved by the library's SM copies between page-locked host memory and the device
    arena, (q_host, o_host, lse_host) = host_buffers(qps, dec.q, dec.o, dec.lse)
    q_host.copy_(dec.q.cpu())
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_bounds = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e0.record(stream)
    for i in range(K):
        qps.copy_host(dec.q, q_host, stream)
        dec.step(stream)
        qps.copy_host(o_host, dec.o, stream)
        qps.copy_host(lse_host, dec.lse, stream)
        e_bounds[i].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    check_device(qps, "the end-to-end steps")
    e2e_ms = max_over_ranks(torch, e0.elapsed_time(e1) / K, world, device)
    e2e_per_step = [e0.elapsed_time(e_bounds[0])] + [e_bounds[i - 1].elapsed_time(e_bounds[i]) for i in range(1, K)]
    o_host, lse_host = o_host.clone(), lse_host.clone()
    arena.close()
    if dec.ring is not None:
        dec.ring.sync()
    return {"step_ms": step_ms, "window_step_ms": window_step_ms, "win_launch_ms": statistics.mean(win_ms),
            "win_launch_p50_ms": statistics.median(win_ms), "per_step": step_distribution(per_step),
            "launches": launches, "clocks": clk, "e2e_ms": e2e_ms, "e2e_per_step": step_distribution(e2e_per_step),
            "h2d": q_host.numel() * q_host.element_size(),
            "d2h": o_host.numel() * o_host.element_size() + lse_host.numel() * lse_host.element_size(),
            "o_host": o_host, "lse_host": lse_host}


def host_buffers(qps, *like):
    """Page-locked, device-mapped host tensors shaped like the given device tensors, in
    one library host arena (returned with them; close it when done)."""
    arena = qps.HostArena(sum(t.numel() * t.element_size() + 256 for t in like))
    return arena, tuple(arena.take(t.shape, t.dtype) for t in like)


def _copy_args(a):
    """An independent copy of an AttnArgs struct (its Python-side references stay with
    the original, which must outlive the copy)."""
    return type(a).from_buffer_copy(a)


def time_window_rotating(torch, qps, args_list, rows, d, stream, n=48):
    """Mean duration of back-to-back window launches that cycle through ``args_list``
    (distinct layers' windows, so that no launch finds the previous one's KV in L2)."""
    n_split = max(qps.attn_plan(a)[0] for a in args_list)
    dev = torch.device("cuda", torch.cuda.current_device())
    parts = (torch.empty((n_split, rows, d), device=dev), torch.empty((n_split, rows), device=dev))
    copies = [_copy_args(a) for a in args_list]
    for a in copies[:3]:
        qps.attn_decode_window(a, parts=parts, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        qps.attn_decode_window(copies[i % len(copies)], parts=parts, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def split_record(torch, qps, synth, cfg, args, dec, m, link_gbs, host_memcpy_gbs, peak, peak_kind, stream,
                 world, ring_plan=None):
    """The figures of one split workload's measurement ``m``."""
    window_bytes, tail_bytes = dec.window_bytes(), dec.tail_bytes()
    kv_bytes = window_bytes + tail_bytes
    L = cfg.layers
    rows = dec.rows
    rec = {"value": whole_job_rate(world, kv_bytes, m["step_ms"]), "unit": UNIT, "ms_per_step": m["step_ms"],
           "dtype": ("f16" if cfg.k_fmt == "f16" and cfg.v_fmt == "f16" else f"{cfg.k_fmt}/{cfg.v_fmt}") +
                    (f" window, {cfg.tk_fmt}/{cfg.tv_fmt} tail" if cfg.mixed else ""),
           "config": bench_config(cfg, args, ring_plan)}
    if dec.window_args:
        n_split_w = qps.attn_plan(dec.window_args[0])[0]
        algo = window_bytes / L + rows * cfg.d * 2 + n_split_w * rows * (cfg.d + 1) * 4
        achieved = algo / (m["win_launch_ms"] / 1e3) / 1e9
        rec["roofline"] = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                           "frac": achieved / peak, "traffic": committed_traffic(traffic_workload(cfg, synth.CONFIGS)),
                           "kernel": "window decode attention (one launch per layer), inside the step",
                           "algorithmic_bytes_per_launch": algo, "launch_ms": m["win_launch_ms"],
                           "launch_p50_ms": m["win_launch_p50_ms"], "n_split": n_split_w,
                           "peak_source": peak_kind}
        # the same launches alone: back to back, cycling through the layers' windows
        iso_ms = time_window_rotating(torch, qps, dec.window_args, rows, cfg.d, stream)
        check_device(qps, "the isolated window launches")
        iso = algo / (iso_ms / 1e3) / 1e9
        rec["roofline_isolated"] = {"bound": "hbm", "achieved": iso, "peak": peak, "unit": "GB/s",
                                    "frac": iso / peak, "launch_ms": iso_ms,
                                    "kernel": "window decode attention alone (48 back-to-back launches "
                                              "cycling through the layers' windows: no L2 reuse)",
                                    "peak_source": peak_kind}
    tail_dma_ms = tail_bytes / (link_gbs * 1e9) * 1e3
    bound_ms = max(m["window_step_ms"], tail_dma_ms)
    if tail_bytes:
        rec["roofline_tail"] = {"bound": "host link", "achieved": tail_bytes / (m["step_ms"] / 1e3) / 1e9,
                                "peak": link_gbs, "unit": "GB/s",
                                "frac": tail_bytes / (m["step_ms"] / 1e3) / 1e9 / link_gbs,
                                "kernel": ("ring copy kernel" if args.ring_copy == "kernel" else "copy engine") +
                                          " (tail tiles, pinned host -> ring slot)",
                                "achieved_source": "tail bytes per step / step time",
                                "peak_source": "pinned 1 GiB host-to-device cudaMemcpyAsync, best of 4, this run"}
    rec["step"] = {"ms": m["step_ms"], "window_only_ms": m["window_step_ms"], "tail_dma_ms": tail_dma_ms,
                   "bound_ms": bound_ms, "ratio_to_bound": m["step_ms"] / bound_ms,
                   "tail_stream_gbs": tail_bytes / (m["step_ms"] / 1e3) / 1e9,
                   "window_only_gbs": window_bytes / (m["window_step_ms"] / 1e3) / 1e9,
                   "link_probe_gbs": link_gbs, "host_memcpy_1thread_gbs": host_memcpy_gbs,
                   "steps_per_s": 1000.0 / m["step_ms"], "per_step": m["per_step"]}
    rec["e2e"] = {"value": whole_job_rate(world, kv_bytes, m["e2e_ms"]), "unit": UNIT,
                  "h2d_bytes_per_step": m["h2d"], "d2h_bytes_per_step": m["d2h"], "ms_per_step": m["e2e_ms"],
                  "per_step": m["e2e_per_step"]}
    rec["gpu_launches"] = m["launches"]
    rec["clocks"] = m["clocks"]
    return rec


def gpu_outputs_of(m, cfg):
    """(O, lse) host arrays of one layer from the last end-to-end step's host buffers."""
    def get(layer):
        return m["o_host"][layer].numpy(), m["lse_host"][layer].numpy()
    return get


def run_split(torch, qps, synth, cfg, args, device, stream, world, rank, gpu_id, link, peak, peak_kind,
              val_layers, cpu_baseline: bool, ring_plan=None):
    dec = build_split(torch, qps, synth, cfg, args, device, n_q=args.n_q)
    try:
        m = time_split_steps(torch, qps, dec, args.steps, args.warmup, stream, world, device, gpu_id)
        rec = split_record(torch, qps, synth, cfg, args, dec, m, link[0], link[1], peak, peak_kind, stream, world,
                           ring_plan)
    finally:
        dec.close()
        del dec
        torch.cuda.empty_cache()
    if rank == 0 and args.n_q == 1 and val_layers:
        b, s, sample, par = time_oracle(cfg, val_layers, device=device, gpu_outputs=gpu_outputs_of(m, cfg))
        rec["validation"] = dict(par, against="float64 CPU oracle on the same seeded inputs",
                                 outputs="last end-to-end step")
        if cpu_baseline:
            rec["cpu_baseline"] = {"value": b / s / 1e9, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                                   "sample": sample + f"; CPU {cpu_model()}"}
    return rec


def run_fanout(torch, qps, synth, cfg, args, device, stream, world, rank, gpu_id, peak, peak_kind):
    """The shared-prefix fan-out as a whole step: one compressed prefix read once for
    every agent, private fp16 suffixes, the per-agent LSE combine; q in, (O, lse) out."""
    import numpy as np

    from quantized_position_split_gb300.decode import FanoutDecoder

    signs = _lib_signs(qps, synth, cfg)
    q = synth.randn_f16((cfg.agents, cfg.hq, cfg.d), cfg.seed, cfg.name, "q", device=device)
    pk = synth.randn_f16((cfg.n_kv, cfg.hkv, cfg.d), cfg.seed, cfg.name, "prefix", "k", device=device)
    pv = synth.randn_f16((cfg.n_kv, cfg.hkv, cfg.d), cfg.seed, cfg.name, "prefix", "v", device=device)
    sk = synth.randn_f16((cfg.agents, cfg.suffix_len, cfg.hkv, cfg.d), cfg.seed, cfg.name, "suffix", "k",
                         device=device)
    sv = synth.randn_f16((cfg.agents, cfg.suffix_len, cfg.hkv, cfg.d), cfg.seed, cfg.name, "suffix", "v",
                         device=device)
    fd = FanoutDecoder(agents=cfg.agents, hq=cfg.hq, hkv=cfg.hkv, d=cfg.d, k_fmt=cfg.k_fmt, v_fmt=cfg.v_fmt,
                       scale=cfg.scale, softcap=cfg.softcap, signs=signs).load(q, pk, pv, sk, sv).build()
    K, W = args.steps, args.warmup
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # > L2: evicts the KV between steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for _ in range(W):
        flush.fill_(0)
        fd.step(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu_id)
    time.sleep(0.3)
    qps.launch_count(reset=True)
    torch.cuda.nvtx.range_push("qps_fanout_timed")  # lets a profiler select the timed launches
    for i in range(K):
        flush.fill_(i & 255)
        ev[i][0].record(stream)
        fd.step(stream)
        ev[i][1].record(stream)
    torch.cuda.nvtx.range_pop()
    launches = qps.launch_count()
    torch.cuda.synchronize()
    clk = clocks.stop()
    check_device(qps, "the timed fan-out steps")
    per_step = [a.elapsed_time(b) for a, b in ev]
    step_ms = max_over_ranks(torch, statistics.mean(per_step), world, device)
    # end to end: q from page-locked host memory in, (O, lse) out, every step (SM copies)
    arena, (q_host, o_host, lse_host) = host_buffers(qps, fd.q, fd.o, fd.lse)
    q_host.copy_(fd.q.cpu())
    e2e = []
    for i in range(K):
        flush.fill_(i & 255)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        qps.copy_host(fd.q, q_host, stream)
        fd.step(stream)
        qps.copy_host(o_host, fd.o, stream)
        qps.copy_host(lse_host, fd.lse, stream)
        b.record(stream)
        e2e.append((a, b))
    torch.cuda.synchronize()
    check_device(qps, "the end-to-end fan-out steps")
    e2e_ms = max_over_ranks(torch, statistics.mean(a.elapsed_time(b) for a, b in e2e), world, device)
    prefix, suffix = fd.prefix_bytes(), fd.suffix_bytes()
    read_once = prefix + suffix
    naive = cfg.agents * prefix + suffix
    rows = cfg.agents * cfg.hq
    n_parts = qps.attn_plan(fd.pre)[0] + qps.attn_plan(fd.suf)[0]
    algo = read_once + rows * cfg.d * 2 + n_parts * rows * (cfg.d + 1) * 4 * 2 + rows * (cfg.d + 1) * 4
    achieved = algo / (step_ms / 1e3) / 1e9
    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "fanout_prefix_traffic.json")) as f:
            tj = json.load(f)
        if tj.get("kernel_source_sha") == attention_source_sha():
            traffic = tj.get("dram_bytes_per_step")
    except (OSError, ValueError):
        pass
    rec = {"value": whole_job_rate(world, read_once, step_ms), "unit": UNIT, "ms_per_step": step_ms,
           "dtype": f"{cfg.k_fmt}/{cfg.v_fmt} prefix, f16 suffixes", "config": bench_config(cfg, args),
           "bytes": {"prefix_read_once": prefix, "suffixes": suffix, "read_once_total": read_once,
                     "naive_per_agent_prefix_reads": naive,
                     "naive_equivalent_gbs": naive / (step_ms / 1e3) / 1e9},
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                        "frac": achieved / peak, "traffic": traffic,
                        "kernel": "whole fan-out step (prefix part, suffix part, combine), L2 flushed before",
                        "algorithmic_bytes_per_step": algo, "peak_source": peak_kind},
           "step": {"ms": step_ms, "per_step": step_distribution(per_step), "steps_per_s": 1000.0 / step_ms},
           "e2e": {"value": whole_job_rate(world, read_once, e2e_ms), "unit": UNIT,
                   "h2d_bytes_per_step": q_host.numel() * q_host.element_size(),
                   "d2h_bytes_per_step": o_host.numel() * o_host.element_size() + lse_host.numel() * 4,
                   "ms_per_step": e2e_ms},
           "gpu_launches": launches, "clocks": clk}
    if rank == 0:
        from oracle import pipeline
        c = lambda t: t.cpu().numpy()  # noqa: E731
        t0 = time.perf_counter()
        ro, rl = pipeline.fanout_reference(c(q), c(pk), c(pv), c(sk), c(sv), cfg.k_fmt, cfg.v_fmt, cfg.scale,
                                           cfg.softcap, _oracle_signs(synth, cfg))
        secs = time.perf_counter() - t0
        par = merge_parity([parity_figures(o_host.numpy(), lse_host.numpy(), ro.reshape(-1, cfg.d), rl.reshape(-1))])
        rec["validation"] = dict(par, against="float64 CPU oracle on the same seeded inputs",
                                 outputs="last end-to-end step", oracle_s=secs)
    del fd, flush
    torch.cuda.empty_cache()
    return rec


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

    qbuild.build()
    qps.device_status(reset=True)
    cfg = line_workload(synth, args)
    if cfg.kind != "split":
        raise SystemExit("the benchmark line times a position-split workload (the fan-out is a sub-record)")
    ring_plan = None
    if args.auto_ring:
        from quantized_position_split_gb300 import autosize
        signs = _lib_signs(qps, synth, cfg)
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

    link = measure_link(torch, device)
    stream = torch.cuda.current_stream()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        gpu_id = None
    peak, peak_kind = measured_hbm_peak()
    # the oracle sample of the main workload: its timing is the cpu_baseline (rank 0 at
    # N = 1); at N > 1 rank 0 still checks one layer of its replica
    main_layers = oracle_layers_for(cfg, args.cpu_layers) if world == 1 else [cfg.layers - 1]
    failed = None
    try:
        main = run_split(torch, qps, synth, cfg, args, device, stream, world, rank, gpu_id, link, peak, peak_kind,
                         main_layers, cpu_baseline=(world == 1 and not args.no_cpu_baseline), ring_plan=ring_plan)
        subs = {}
        for name in [s for s in args.sub_configs.split(",") if s.strip()]:
            sc = synth.by_name(name.strip())
            if sc.name == cfg.name:
                continue
            if sc.kind == "fanout":
                subs[sc.name] = run_fanout(torch, qps, synth, sc, args, device, stream, world, rank, gpu_id, peak,
                                           peak_kind)
            else:
                val = [sc.layers - 1] if sc.d > 128 or world > 1 else [0, sc.layers - 1]
                subs[sc.name] = run_split(torch, qps, synth, sc, args, device, stream, world, rank, gpu_id, link,
                                          peak, peak_kind, val, cpu_baseline=False)
    except DeviceCheckFailed as e:
        failed = str(e)
    if failed:
        print(f"bench.py: {failed}; the figures of this run are not valid", file=sys.stderr, flush=True)
        return 3
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    out = {
        "metric": METRIC,
        "value": main["value"],
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": main["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": main["dtype"],
        "data": DATA,
        "config": main["config"],
        "roofline": main["roofline"],
        "roofline_isolated": main.get("roofline_isolated"),
        "roofline_tail": main.get("roofline_tail"),
        "step": main["step"],
        "cpu_baseline": main.get("cpu_baseline"),
        "validation": main.get("validation"),
        "e2e": main["e2e"],
        "gpu_launches": main["gpu_launches"],
        "clocks": main["clocks"],
        "sub_records": subs,
    }
    print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    bad = [n for n, r in [(cfg.name, main)] + list(subs.items())
           if r.get("validation") is not None and not r["validation"]["pass"]]
    if bad:
        print(f"bench.py: outputs outside the parity bar for {bad}", file=sys.stderr, flush=True)
        return 4
    return 0


# kernel-only lines of a workload's window with (K, V) stored in other formats: V at the
# other TurboQuant tiers, and K and V both TurboQuant (K read in the rotated domain)
TIER_VARIANTS = {"qwen14b_q8": (("q8_0", "tq4"), ("q8_0", "tq2"), ("tq4", "tq4"), ("tq3", "tq3"), ("tq2", "tq2")),
                 "gemma_global_q8k_tq3v": (("q8_0", "tq4"), ("q8_0", "tq2"), ("tq3", "tq3"))}


def run_kernel_only(args):
    """Per-launch time of the window decode-attention kernel on one layer of each
    workload (or of --config), timed back to back with CUDA events.  The launches cycle
    through enough copies of the window (each at its own address) that together they
    exceed 3 x L2, so no launch reads the previous one's KV from L2; the fan-out
    prefix is flagged as L2-sized."""
    import torch

    import synth
    import quantized_position_split_gb300 as qps
    from quantized_position_split_gb300 import build as qbuild

    qbuild.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    # (the mixed-tail workloads share their window kernel with the uniform ones)
    names = [args.config] if args.config != DEFAULT_CONFIG or args.layers else [
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
            shared = False
            rows = cfg.batch * cfg.hq
        else:
            q = synth.randn_f16((cfg.agents, cfg.hq, cfg.d), cfg.seed, cfg.name, "q", device=dev)
            k = synth.randn_f16((cfg.n_kv, cfg.hkv, cfg.d), cfg.seed, cfg.name, "prefix", "k", device=dev)
            v = synth.randn_f16((cfg.n_kv, cfg.hkv, cfg.d), cfg.seed, cfg.name, "prefix", "v", device=dev)
            shared = True
            rows = cfg.agents * cfg.hq

        def windows(kf, vf, qq, **kw):
            first = (qps.encode_kv_head_major(kf, k, signs), qps.encode_kv_head_major(vf, v, signs))
            kvb = first[0].nbytes() + first[1].nbytes()
            n_copies = 1 if cfg.kind != "split" else max(1, min(8, math.ceil(3 * L2_BYTES / kvb)))
            kvs = [first] + [(qps.encode_kv_head_major(kf, k, signs), qps.encode_kv_head_major(vf, v, signs))
                             for _ in range(n_copies - 1)]
            return kvs, [qps.attn_args(qq, K, V, scale=cfg.scale, softcap=cfg.softcap, v_signs=signs,
                                       shared=shared, **kw) for K, V in kvs]

        variants = [(cfg.k_fmt, cfg.v_fmt, 1)]
        if name == DEFAULT_CONFIG and cfg.kind == "split":
            variants.append((cfg.k_fmt, cfg.v_fmt, 4))
        if not (args.layers or args.v_fmt or args.k_fmt):
            variants += [(kf, vf, 1) for kf, vf in TIER_VARIANTS.get(name, ())]
        for kf, vf, n_q in variants:
            if n_q > 1:  # a verify batch: 4 query tokens at the end of the window, causal
                qq = synth.randn_f16((cfg.batch, n_q, cfg.hq, cfg.d), cfg.seed, cfg.name, "verify", device=dev)
                kvs, alist = windows(kf, vf, qq, q_pos=cfg.wc - n_q)
                label = f"{name} verify n_q={n_q} causal"
            else:
                kvs, alist = windows(kf, vf, q)
                label = name if (kf, vf) == (cfg.k_fmt, cfg.v_fmt) else f"{name} K={kf} V={vf}"
            r = rows * n_q
            us = time_window_rotating(torch, qps, alist, r, cfg.d, s, n=50) * 1e3
            n_split = qps.attn_plan(alist[0])[0]
            kv = kvs[0][0].nbytes() + kvs[0][1].nbytes()
            algo = kv + r * cfg.d * 2 + n_split * r * (cfg.d + 1) * 4
            print(json.dumps({"kernel": "attn_decode_window", "workload": label, "path": qps.attn_path(alist[0]),
                              "n_split": n_split, "launch_us": us, "kv_bytes": kv, "algorithmic_bytes": algo,
                              "achieved_gbs": algo / us / 1e3, "frac_of_hbm": algo / us / 1e3 / peak,
                              "peak_gbs": peak, "peak_source": peak_kind, "window_copies": len(kvs),
                              "l2_resident": kv < L2_BYTES and len(kvs) == 1}), flush=True)
            del kvs, alist
        qps.device_status(reset=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel_only:
        return run_kernel_only(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
