"""Measured ring sizing and storage-tier choice for a position-split decode.

The auto-adapt loop of "F5 M7 — Rolling KV: position-windowed KV residency" (section
"Auto-adapt loop"): measure the host link, from pinned host memory through the copy
engine — the path every tail tile takes, so the figure already includes whatever host
RAM can feed it ("T*-aware auto rolling-KV spill", section "T* — the negligible-drop
tail band", bounds the link by host RAM bandwidth; a CPU copy would measure the cores,
not the RAM the copy engine reads, and is only reported), time one layer's attention at
the target context on
this GPU, measure the fixed cost of engaging the streamed tail ("c_engage boot probe":
the same layer resident, and with a small tail streamed through the ring), then let
the library's policy calls size the ring (qps_plan_ring), the tail band T*
(qps_tail_band) and the storage tier (qps_choose_tier).  Every measurement runs the
library's own kernels and ring on synthetic data of the workload's shapes.
"""

from __future__ import annotations

import time
from typing import Optional, Sequence, Tuple

import torch

from . import (Ring, attn_args, attn_decode_window, attn_plan, choose_tier, encode_kv_head_major, lse_combine,
               plan_ring, plane_row_bytes, tail_band, tile_desc)


def measure_link(device, nbytes: int = 256 << 20, reps: int = 3) -> Tuple[float, float]:
    """(pinned host -> device GB/s, host RAM copy GB/s), best of ``reps``.  The host
    figure is a copy spread over the process's CPU threads (torch's parallel copy): the
    copy engine reads host RAM directly, so a single thread's rate would understate
    what RAM can feed the link."""
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dev = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s = torch.cuda.current_stream(device)
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        dev.copy_(host, non_blocking=True)
        e1.record(s)
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    link = nbytes / (best * 1e-3) / 1e9
    a = torch.ones(nbytes, dtype=torch.uint8)
    b = torch.empty_like(a)
    t_best = float("inf")
    for _ in range(reps):
        t0 = time.perf_counter()
        b.copy_(a)
        t_best = min(t_best, time.perf_counter() - t0)
    return link, nbytes / t_best / 1e9


def _layer_kv(n, hkv, d, device, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    k = torch.randn((n, hkv, d), generator=g).half().to(device)
    v = torch.randn((n, hkv, d), generator=g).half().to(device)
    return k, v


def _time(fn, reps, device):
    s = torch.cuda.current_stream(device)
    for _ in range(3):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record(s)
    for _ in range(reps):
        fn()
    e1.record(s)
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1) / reps


def attention_ms(k_fmt: str, v_fmt: str, *, batch: int, hq: int, hkv: int, d: int, n_kv: int, scale: float,
                 softcap: float = 0.0, signs=None, device=None, reps: int = 20) -> float:
    """One layer's decode attention over ``n_kv`` device-resident positions (ms)."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    k, v = _layer_kv(n_kv, hkv, d, device, 11)
    K, V = encode_kv_head_major(k_fmt, k, signs), encode_kv_head_major(v_fmt, v, signs)
    del k, v
    q = torch.randn((batch, hq, d), device=device).half()
    a = attn_args(q, K, V, scale=scale, softcap=softcap, v_signs=signs)
    o = torch.empty((batch * hq, d), device=device)
    lse = torch.empty((batch * hq,), device=device)
    return _time(lambda: attn_decode_window(a, o=o, lse=lse), reps, device)


def c_engage_ms(k_fmt: str, v_fmt: str, *, batch: int, hq: int, hkv: int, d: int, n_kv: int, scale: float,
                softcap: float = 0.0, signs=None, device=None, tail_tokens: int = 256, reps: int = 20) -> float:
    """The fixed per-layer cost of engaging the streamed tail: the same layer with a
    ``tail_tokens`` tail streamed through a two-slot ring, minus fully resident (ms,
    never below 0)."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    wc = n_kv - tail_tokens
    k, v = _layer_kv(n_kv, hkv, d, device, 12)
    K, V = encode_kv_head_major(k_fmt, k, signs), encode_kv_head_major(v_fmt, v, signs)
    Kw, Vw = encode_kv_head_major(k_fmt, k[:wc], signs), encode_kv_head_major(v_fmt, v[:wc], signs)
    Kt = encode_kv_head_major(k_fmt, k[wc:], signs).pinned_copy()
    Vt = encode_kv_head_major(v_fmt, v[wc:], signs).pinned_copy()
    del k, v
    q = torch.randn((batch, hq, d), device=device).half()
    full = attn_args(q, K, V, scale=scale, softcap=softcap, v_signs=signs)
    o = torch.empty((batch * hq, d), device=device)
    lse = torch.empty((batch * hq,), device=device)
    t_res = _time(lambda: attn_decode_window(full, o=o, lse=lse), reps, device)

    win = attn_args(q, Kw, Vw, scale=scale, softcap=softcap, v_signs=signs)
    tail = attn_args(q, Kt, Vt, scale=scale, softcap=softcap, v_signs=signs)
    nw, nt = attn_plan(win)[0], attn_plan(tail)[0]
    parts = (torch.empty((nw + nt, batch * hq, d), device=device), torch.empty((nw + nt, batch * hq), device=device))
    td = tile_desc(Kt, Vt)
    need = sum((x + 255) // 256 * 256 for x in list(td.bytes_k) + list(td.bytes_v))
    ring = Ring(2, need, device.index)

    def windowed():
        attn_decode_window(win, parts=parts, part_offset=0)
        ring.begin_step([td])
        ring.decode_tail(0, tail, parts=parts, part_offset=nw)
        ring.end_step()
        lse_combine(parts[0], parts[1], o=o, lse=lse)

    t_win = _time(windowed, reps, device)
    ring.sync()
    ring.close()
    return max(0.0, t_win - t_res)


def plan_decode(*, layers: int, batch: int, hq: int, hkv: int, d: int, n_kv: int,
                tiers: Sequence[Tuple[str, str]], device_budget_bytes: float, scale: float,
                softcap: float = 0.0, signs=None, w_active_bytes: float = 0.0, vram_gbs: Optional[float] = None,
                target_drop: float = 0.20, device=None, measured: Optional[dict] = None) -> dict:
    """Storage tier, window length and ring shape for a ``layers``-layer cache.

    ``tiers`` lists (k_fmt, v_fmt) from least to most compressing.  The tier is the
    first whose whole cache fits ``device_budget_bytes`` + T*; the window keeps as many
    positions as the budget holds (rounded down to 16), the tail the rest, streamed in
    tiles sized by ``plan_ring`` from the measured link and attention time, in ring
    slots paid from what the window leaves of the budget.  ``measured`` may supply the
    link / host-copy / attention / engagement figures instead of measuring them.
    """
    m = dict(measured or {})

    def dev():  # only the measurements touch the GPU
        return device or torch.device("cuda", torch.cuda.current_device())

    if "link_gbs" not in m or "host_memcpy_gbs" not in m:
        m["link_gbs"], m["host_memcpy_gbs"] = measure_link(dev())
    bw_eff = m["link_gbs"]
    if vram_gbs is None:
        vram_gbs = m.get("vram_gbs", 6000.0)

    def per_token(fmt_k, fmt_v):  # stored bytes of one position of one layer
        def row(fmt):
            return sum(plane_row_bytes(fmt, d))
        return hkv * (row(fmt_k) + row(fmt_v))

    kv_bytes = [layers * n_kv * per_token(kf, vf) for kf, vf in tiers]
    t_res = (w_active_bytes + kv_bytes[0]) / (vram_gbs * 1e9) * 1e3
    if "c_engage_ms" not in m:
        kf, vf = tiers[0]
        m["c_engage_ms"] = layers * c_engage_ms(kf, vf, batch=batch, hq=hq, hkv=hkv, d=d, n_kv=n_kv,
                                                 scale=scale, softcap=softcap, signs=signs, device=dev())
    t_star = tail_band(t_res, m["c_engage_ms"], bw_eff, target_drop)
    tier = choose_tier(kv_bytes, device_budget_bytes, t_star)
    kf, vf = tiers[tier]
    ptb = per_token(kf, vf)
    wc = int(min(n_kv, device_budget_bytes // (layers * ptb)) // 16 * 16)
    tail_tokens = n_kv - wc
    out = dict(m, bw_eff_gbs=bw_eff, vram_gbs=vram_gbs, t_resident_ms=t_res, t_star_bytes=t_star,
               tier=tier, k_fmt=kf, v_fmt=vf, wc=wc, tail_tokens=tail_tokens,
               tail_bytes=float(layers * tail_tokens * ptb), kv_bytes_per_tier=kv_bytes)
    if tail_tokens == 0:
        out.update(ring_slots=0, tile_tokens=0)
        return out
    if "attention_ms" not in m:
        m["attention_ms"] = attention_ms(kf, vf, batch=batch, hq=hq, hkv=hkv, d=d, n_kv=n_kv, scale=scale,
                                         softcap=softcap, signs=signs, device=dev())
        out["attention_ms"] = m["attention_ms"]
    slot_budget = max(device_budget_bytes - layers * wc * ptb, 1.0)
    ring = plan_ring(m["attention_ms"], bw_eff, slot_budget, float(tail_tokens * ptb))
    tile_tokens = max(16, int(ring["tile_bytes"] // ptb) // 16 * 16)
    tile_tokens = min(tile_tokens, (tail_tokens + 15) // 16 * 16)
    out.update(ring_slots=ring["n_slots"], tile_tokens=tile_tokens, ring=ring)
    return out
