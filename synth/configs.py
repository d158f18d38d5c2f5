"""Workload shapes: the decode configurations and their parity-sized copies.

Every field is a plain shape or format name; nothing here computes anything.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "split" (window + host tail) or "fanout" (shared prefix + private suffixes)
    layers: int
    batch: int
    hq: int
    hkv: int
    d: int
    n_kv: int  # split: total positions; fanout: prefix length
    wc: int  # split: device window length; fanout: unused (= n_kv)
    k_fmt: str  # "f16" | "q8_0" | "tq2" | "tq3" | "tq4" (with V in the same tier)
    v_fmt: str  # "f16" | "q8_0" | "tq2" | "tq3" | "tq4"
    softcap: float = 0.0  # <= 0: off
    tail_k_fmt: Optional[str] = None  # split: the tail's K format (None: k_fmt)
    tail_v_fmt: Optional[str] = None  # split: the tail's V format (None: v_fmt)
    k_outliers: int = 0  # channels per (layer, KV head) scaled by outlier_scale
    outlier_scale: float = 20.0
    ring_slots: int = 3
    tile_tokens: int = 8192
    agents: int = 0  # fanout: number of agents sharing the prefix
    suffix_len: int = 0  # fanout: private fp16 suffix per agent
    sign_seed: int = 42
    sign_seed2: Optional[int] = None  # TurboQuant second sign vector (None: none)
    rot_block: int = 0  # TurboQuant Hadamard block width (0: head_dim)
    seed: int = 1234

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    @property
    def tk_fmt(self) -> str:
        return self.k_fmt if self.tail_k_fmt is None else self.tail_k_fmt

    @property
    def tv_fmt(self) -> str:
        return self.v_fmt if self.tail_v_fmt is None else self.tail_v_fmt

    @property
    def mixed(self) -> bool:
        return (self.tk_fmt, self.tv_fmt) != (self.k_fmt, self.v_fmt)

    @property
    def tail_len(self) -> int:
        return self.n_kv - self.wc if self.kind == "split" else 0

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


CONFIGS = [
    Workload(
        name="tiny",
        kind="split",
        layers=1,
        batch=1,
        hq=4,
        hkv=1,
        d=64,
        n_kv=1024,
        wc=512,
        k_fmt="f16",
        v_fmt="f16",
        ring_slots=2,
        tile_tokens=256,
    ),
    Workload(
        name="qwen14b_f16",
        kind="split",
        layers=48,
        batch=1,
        hq=40,
        hkv=8,
        d=128,
        n_kv=65536,
        wc=32768,
        k_fmt="f16",
        v_fmt="f16",
        k_outliers=4,
        ring_slots=3,
        tile_tokens=32768,
    ),
    Workload(
        name="qwen14b_q8",
        kind="split",
        layers=48,
        batch=1,
        hq=40,
        hkv=8,
        d=128,
        n_kv=131072,
        wc=98304,
        k_fmt="q8_0",
        v_fmt="q8_0",
        k_outliers=4,
        ring_slots=3,
        tile_tokens=32768,
    ),
    Workload(
        name="gemma_global_q8k_tq3v",
        kind="split",
        layers=5,
        batch=1,
        hq=16,
        hkv=2,
        d=512,
        n_kv=262144,
        wc=131072,
        k_fmt="q8_0",
        v_fmt="tq3",
        softcap=50.0,
        k_outliers=4,
        ring_slots=3,
        tile_tokens=131072,
    ),
    # the same Qwen-like stacks with a more compressed tail than window (the tail's own
    # K / V storage formats)
    Workload(
        name="qwen14b_f16_q8tail",
        kind="split",
        layers=48,
        batch=1,
        hq=40,
        hkv=8,
        d=128,
        n_kv=65536,
        wc=32768,
        k_fmt="f16",
        v_fmt="f16",
        tail_k_fmt="q8_0",
        tail_v_fmt="q8_0",
        k_outliers=4,
        ring_slots=3,
        tile_tokens=16384,
    ),
    Workload(
        name="qwen14b_q8_tq3vtail",
        kind="split",
        layers=48,
        batch=1,
        hq=40,
        hkv=8,
        d=128,
        n_kv=131072,
        wc=98304,
        k_fmt="q8_0",
        v_fmt="q8_0",
        tail_k_fmt="q8_0",
        tail_v_fmt="tq3",
        k_outliers=4,
        ring_slots=3,
        tile_tokens=16384,
    ),
    # the smallest tail: V at the 2-bit TurboQuant tier
    Workload(
        name="qwen14b_q8_tq2vtail",
        kind="split",
        layers=48,
        batch=1,
        hq=40,
        hkv=8,
        d=128,
        n_kv=131072,
        wc=98304,
        k_fmt="q8_0",
        v_fmt="q8_0",
        tail_k_fmt="q8_0",
        tail_v_fmt="tq2",
        k_outliers=4,
        ring_slots=3,
        tile_tokens=16384,
    ),
    # a tail with K and V both at the 3-bit TurboQuant tier (K read in the rotated domain)
    Workload(
        name="qwen14b_q8_tq3kvtail",
        kind="split",
        layers=48,
        batch=1,
        hq=40,
        hkv=8,
        d=128,
        n_kv=131072,
        wc=98304,
        k_fmt="q8_0",
        v_fmt="q8_0",
        tail_k_fmt="tq3",
        tail_v_fmt="tq3",
        k_outliers=4,
        ring_slots=3,
        tile_tokens=16384,
    ),
    # the Gemma-like global layers with the rotation the pages' fork runs at head_dim 512:
    # four independent 128-wide Hadamard blocks between two sign vectors
    Workload(
        name="gemma_global_q8k_tq3v_r128",
        kind="split",
        layers=5,
        batch=1,
        hq=16,
        hkv=2,
        d=512,
        n_kv=262144,
        wc=131072,
        k_fmt="q8_0",
        v_fmt="tq3",
        softcap=50.0,
        k_outliers=4,
        ring_slots=3,
        tile_tokens=32768,
        sign_seed2=43,
        rot_block=128,
    ),
    Workload(
        name="fanout_prefix",
        kind="fanout",
        layers=1,
        batch=15,
        hq=32,
        hkv=8,
        d=128,
        n_kv=4096,
        wc=4096,
        k_fmt="q8_0",
        v_fmt="tq3",
        agents=15,
        suffix_len=512,
    ),
]


def by_name(name: str) -> Workload:
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


def parity_scaled(cfg: Workload, layers: Optional[int] = None) -> Workload:
    """A copy of ``cfg`` small enough for the float64 oracle to finish in seconds.

    Head counts, head_dim, formats, softcap and (unless ``layers`` is given) the layer
    count are kept; positions are cut to a few thousand with deliberately ragged window
    / tile boundaries so that the GPU path crosses several split chunks, several ring
    tiles and a partial last tile.
    """
    if cfg.kind == "fanout":
        return cfg.replace(n_kv=1000, wc=1000, suffix_len=77, agents=min(cfg.agents, 15))
    n = 3000 + 37 if cfg.d <= 128 else 2000 + 21
    wc = 1101 if cfg.d <= 128 else 777
    return cfg.replace(
        layers=layers if layers is not None else cfg.layers,
        n_kv=n,
        wc=wc,
        tile_tokens=512,
    )
