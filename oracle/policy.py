"""Residency and ring sizing policy (oracle; test infrastructure only).

Plain float64 arithmetic of three passages:

* "F5 M7 — Rolling KV: position-windowed KV residency", section "Slot pool": the largest
  tile the link can move while one layer's attention runs, with a 0.8 safety factor,
  and 2..4 slots from the device budget; section "Auto-adapt loop": a layer's tail
  larger than one tile runs as several position sub-tiles.
* "T*-aware auto rolling-KV spill (HAL #582 P1+, #621 follow-on)", section "T* — the
  negligible-drop tail band": the per-token drop of streaming a tail and the largest
  tail T* that keeps it under the target; section "The decision (fit-condition
  reformulation)": the first (least compressing) storage tier whose bytes fit the
  device budget plus T*, else the most compressing one.

Readings where the pages are silent: slots are whole numbers (the quotient is floored
before the clamp); a layer's tail is cut into the fewest equal tiles no larger than the
maximum; T* below zero means "never spill" and is reported as 0; bandwidths are in GB/s
(1e9 bytes/s) and times in milliseconds.
"""

from __future__ import annotations

import math


def ring_plan(compute_ms_per_layer: float, bw_eff_gbs: float, slot_budget_bytes: float,
              per_layer_tail_bytes: float, safety: float = 0.8):
    """(n_slots, tiles_per_layer, tile_bytes, tile_bytes_max) of the prefetch ring."""
    tile_bytes_max = compute_ms_per_layer * 1e-3 * bw_eff_gbs * 1e9 * safety
    n_slots = int(min(4, max(2, math.floor(slot_budget_bytes / tile_bytes_max))))
    if per_layer_tail_bytes <= 0:
        return n_slots, 0, 0, tile_bytes_max
    tiles = int(math.ceil(per_layer_tail_bytes / tile_bytes_max))
    tile_bytes = int(math.ceil(per_layer_tail_bytes / tiles))
    return n_slots, tiles, tile_bytes, tile_bytes_max


def t_resident_ms(w_active_bytes: float, kv_resident_bytes: float, vram_bw_gbs: float) -> float:
    """Per-token time with the whole cache resident: every active byte read once."""
    return (w_active_bytes + kv_resident_bytes) / (vram_bw_gbs * 1e9) * 1e3


def tail_drop(c_engage_ms: float, tail_bytes: float, bw_eff_gbs: float, t_resident: float) -> float:
    """Fractional per-token slowdown of streaming ``tail_bytes`` from the host."""
    return (c_engage_ms + tail_bytes / (bw_eff_gbs * 1e9) * 1e3) / t_resident


def t_star_bytes(t_resident: float, c_engage_ms: float, bw_eff_gbs: float, target_drop: float = 0.20) -> float:
    """The largest tail whose drop stays at ``target_drop`` (0: never spill)."""
    t = (target_drop * t_resident - c_engage_ms) * 1e-3 * bw_eff_gbs * 1e9
    return max(0.0, t)


def choose_tier(kv_bytes_per_tier, budget_bytes: float, t_star: float) -> int:
    """Index of the first tier (least to most compressing) with bytes <= budget + T*;
    the last tier when none fits (the rolling window spills the rest)."""
    for i, b in enumerate(kv_bytes_per_tier):
        if b <= budget_bytes + t_star:
            return i
    return len(kv_bytes_per_tier) - 1
