"""Assembly of a whole position-split decode step from per-layer fp16 K / V caches.

Each layer's cache is encoded on the GPU by the library's encoders.  Its window
[0, wc) stays in device memory; its tail [wc, n_kv) is cut into tiles of
``tile_tokens`` positions, each copied once to pinned host memory as one contiguous
range per plane ("Rolling-KV: step/graph-level tail prefetch (design)", section "The
fix: a persistent, step-spanning tail-prefetch ring"; "F5 M7 — Rolling KV:
position-windowed KV residency", header status block).  Both are stored head-major
(consecutive positions of one KV head are adjacent rows, head length padded to 16) so
that the tensor-core decode streams each head's rows as one range.  A step is one
``qps_decode_step`` call: per layer, the window part, the layer's ring tiles, and the
LSE combine.

The shared-prefix batch ("F5 M6 — PolyKV (shared compressed KV pool)", section "S1 —
SharedKVPool") is assembled by ``FanoutDecoder``: one compressed prefix read by every
agent in one pass, plus one private fp16 suffix per agent, merged per agent.
"""

from __future__ import annotations

from typing import List, Optional

import torch

from . import KV, HostArena, Ring, StepPlan, attn_args, attn_plan, encode_kv_head_major, plane_row_bytes, tile_desc


def _parts_buffers(capacity: int, rows: int, d: int, device):
    return (torch.empty((capacity, rows, d), dtype=torch.float32, device=device),
            torch.empty((capacity, rows), dtype=torch.float32, device=device))


class PositionSplitDecoder:
    """Decode attention of ``layers`` layers over a KV cache split at ``wc``.

    ``tail_k_fmt`` / ``tail_v_fmt`` store the tail in other (normally more compressed)
    formats than the window ("F5 M7 — Rolling KV: position-windowed KV residency",
    section "2026-07-12 — #582-P2 SHIPPED: position-axis mixed KV (compressed tail,
    -ctkt/-ctvt)"): the recent positions keep the window's formats on the device, the
    tail ships fewer bytes per step, and each part is read at its own format.  Unset,
    the tail uses the window's formats.

    ``n_q`` > 1 makes each step a verify batch ("F5 M6 — PolyKV", section "S2 perf-path
    — turbo-MMA verify kernel"): q is [batch = 1, n_q, hq, D], the n_q query tokens are
    the cache's last n_q positions, and with ``causal`` token i sees the positions up to
    n_kv - n_q + i (they lie in the tail when the tail is non-empty: each tile carries
    its first position to the ring)."""

    def __init__(self, *, layers: int, batch: int, hq: int, hkv: int, d: int, n_kv: int, wc: int,
                 k_fmt: str, v_fmt: str, scale: float, softcap: float = 0.0, signs=None,
                 ring_slots: int = 3, tile_tokens: int = 0, n_split_window: int = 0,
                 n_split_tail: int = 0, device=None, host_alloc_flags: int = 2,
                 tail_k_fmt: Optional[str] = None, tail_v_fmt: Optional[str] = None,
                 ring_copy: str = "kernel", n_q: int = 1, causal: bool = True):
        if not 0 <= wc <= n_kv:
            raise ValueError("need 0 <= wc <= n_kv")
        if n_q > 1 and batch != 1:
            raise ValueError("a verify batch (n_q > 1) decodes one sequence (batch 1)")
        if not 1 <= n_q <= min(64, max(n_kv, 1)):
            raise ValueError("need 1 <= n_q <= min(64, n_kv)")
        self.n_q = n_q
        self.q_pos = n_kv - n_q if (n_q > 1 and causal) else None
        self.host_alloc_flags = host_alloc_flags
        # "kernel": the ring's copy kernel moves the tail (arena) tiles: the copy engine's
        # host-to-device transfers stall in bursts on some GB300 hosts (steps of 31 ms
        # taking up to 320 ms) where SM loads of the same memory do not; "engine":
        # cudaMemcpyAsync (5% faster when nothing stalls, and no SMs taken)
        self.ring_copy = ring_copy
        self.layers, self.batch, self.hq, self.hkv, self.d = layers, batch, hq, hkv, d
        self.n_kv, self.wc = n_kv, wc
        self.k_fmt, self.v_fmt = k_fmt, v_fmt
        self.tail_k_fmt = k_fmt if tail_k_fmt is None else tail_k_fmt
        self.tail_v_fmt = v_fmt if tail_v_fmt is None else tail_v_fmt
        self.scale, self.softcap, self.signs = scale, softcap, signs
        self.ring_slots, self.tile_tokens = ring_slots, tile_tokens
        self.n_split_window, self.n_split_tail = n_split_window, n_split_tail
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.rows = batch * n_q * hq
        qshape = (layers, batch, hq, d) if n_q == 1 else (layers, batch, n_q, hq, d)
        self.q = torch.zeros(qshape, dtype=torch.float16, device=self.device)
        self.o = torch.zeros((layers, self.rows, d), dtype=torch.float32, device=self.device)
        self.lse = torch.zeros((layers, self.rows), dtype=torch.float32, device=self.device)
        self.window: List[Optional[tuple]] = [None] * layers  # (K, V) on device
        self.tail: List[list] = [[] for _ in range(layers)]  # per tile: (K, V) pinned host
        self.ring: Optional[Ring] = None
        self.arena: Optional[HostArena] = None
        self.plan: Optional[StepPlan] = None
        self.window_plan: Optional[StepPlan] = None

    @property
    def tail_len(self) -> int:
        return self.n_kv - self.wc

    def tile_ranges(self):
        """The tail's ring tiles: ``tile_tokens`` positions each, or with 0 (the default)
        one tile per layer's tail — every copy launch costs the link ~11 us, and on
        GB300 one tile per layer ran the Qwen-like q8_0 step 3% faster than two."""
        t = self.tile_tokens if self.tile_tokens > 0 else max(self.tail_len, 1)
        return [(a, min(a + t, self.tail_len)) for a in range(0, self.tail_len, t)]

    def _arena_bytes(self) -> int:
        """Pinned bytes the whole tail needs: every tile's planes, 256-byte aligned."""
        def plane_bytes(fmt):
            return plane_row_bytes(fmt, self.d)
        total = 0
        for a, b in self.tile_ranges():
            tp = (b - a + 15) // 16 * 16
            for rb in plane_bytes(self.tail_k_fmt) + plane_bytes(self.tail_v_fmt):
                total += (self.hkv * tp * rb + 255) // 256 * 256
        return total * self.layers

    def load_layer(self, layer: int, k16: torch.Tensor, v16: torch.Tensor, q16: Optional[torch.Tensor] = None):
        """Encode one layer's fp16 ``k16, v16[n_kv, hkv, d]`` (CUDA) and place it.

        The tail tiles of every layer share one page-locked arena (``qps_host_alloc``,
        by default backed by transparent huge pages): the copy engine then reads a few
        large pinned regions.  Hundreds of separate pinned allocations showed periodic
        copy stalls of 100+ ms on GB300 hosts."""
        if self.wc > 0:
            self.window[layer] = (encode_kv_head_major(self.k_fmt, k16[:self.wc], self.signs),
                                  encode_kv_head_major(self.v_fmt, v16[:self.wc], self.signs))
        tiles = []
        ranges = self.tile_ranges()
        if ranges and self.arena is None:
            self.arena = HostArena(self._arena_bytes(), self.host_alloc_flags)
        for a, b in ranges:
            kt = encode_kv_head_major(self.tail_k_fmt, k16[self.wc + a:self.wc + b], self.signs)
            vt = encode_kv_head_major(self.tail_v_fmt, v16[self.wc + a:self.wc + b], self.signs)
            tiles.append((self.arena.copy_in(kt), self.arena.copy_in(vt), self.wc + a))
        self.tail[layer] = tiles
        if q16 is not None:
            self.q[layer].copy_(q16)

    def _args(self, layer, k: KV, v: KV, n_split: int):
        return attn_args(self.q[layer], k, v, scale=self.scale, softcap=self.softcap,
                         v_signs=self.signs, n_split=n_split, q_pos=self.q_pos)

    def build(self):
        """Create the ring, the flat (layer, tile) schedule and the step plans."""
        tiles = []
        slot_bytes = 0
        for layer in range(self.layers):
            for kt, vt, pos0 in self.tail[layer]:
                td = tile_desc(kt, vt, pos0=pos0)
                tiles.append(td)
                need = sum((x + 255) // 256 * 256 for x in list(td.bytes_k) + list(td.bytes_v))
                slot_bytes = max(slot_bytes, need)
        if tiles:
            self.ring = Ring(self.ring_slots, slot_bytes, self.device.index, copy=self.ring_copy)
        layers, wlayers = [], []
        self._keep = []
        self.window_args = []
        for layer in range(self.layers):
            parts, cap = [], 0
            if self.window[layer] is not None:
                kw, vw = self.window[layer]
                wargs = self._args(layer, kw, vw, self.n_split_window)
                self.window_args.append(wargs)
                parts.append(wargs)
                cap += attn_plan(wargs)[0]
            tail_tpl = None
            for kt, vt, _ in self.tail[layer]:
                probe = self._args(layer, kt, vt, self.n_split_tail)
                cap += attn_plan(probe)[0]
                if tail_tpl is None:
                    # a template: the ring replaces data pointers and strides with its slot's
                    tail_tpl = probe
            o_parts, lse_parts = _parts_buffers(max(cap, 1), self.rows, self.d, self.device)
            self._keep += [o_parts, lse_parts]
            layers.append(dict(device_parts=parts, tail=tail_tpl, n_tiles=len(self.tail[layer]),
                               o_parts=o_parts, lse_parts=lse_parts, o=self.o[layer], lse=self.lse[layer]))
            if parts:
                wlayers.append(dict(device_parts=parts, tail=None, n_tiles=0, o_parts=o_parts,
                                    lse_parts=lse_parts, o=self.o[layer], lse=self.lse[layer]))
        self.plan = StepPlan(layers, tiles, self.ring)
        self.window_plan = StepPlan(wlayers) if wlayers else None
        self.n_tiles = len(tiles)
        return self

    def step(self, stream=None):
        self.plan.run(stream)

    def window_step(self, stream=None):
        """The same step with the ring and the tail omitted (window parts + combines)."""
        if self.window_plan is not None:
            self.window_plan.run(stream)

    # algorithmic bytes: every stored plane the step must read once
    def window_bytes(self) -> int:
        return sum(kv.nbytes() for w in self.window if w is not None for kv in w)

    def tail_bytes(self) -> int:
        return sum(kv.nbytes() for t in self.tail for tile in t for kv in tile[:2])

    def close(self):
        """Release the ring (after its copies finish), the plans and the host arena."""
        if self.ring is not None:
            self.ring.close()
            self.ring = None
        self.plan = self.window_plan = None
        self.tail = [[] for _ in range(self.layers)]
        if self.arena is not None:
            self.arena.close()
            self.arena = None


class FanoutDecoder:
    """One compressed prefix shared by ``agents`` sets of query rows, plus private fp16
    suffixes; one layer, all device-resident."""

    def __init__(self, *, agents: int, hq: int, hkv: int, d: int, k_fmt: str, v_fmt: str,
                 scale: float, softcap: float = 0.0, signs=None, n_split_prefix: int = 0,
                 n_split_suffix: int = 0, device=None):
        self.agents, self.hq, self.hkv, self.d = agents, hq, hkv, d
        self.k_fmt, self.v_fmt = k_fmt, v_fmt
        self.scale, self.softcap, self.signs = scale, softcap, signs
        self.n_split_prefix, self.n_split_suffix = n_split_prefix, n_split_suffix
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.rows = agents * hq
        self.q = torch.zeros((agents, hq, d), dtype=torch.float16, device=self.device)
        self.o = torch.zeros((self.rows, d), dtype=torch.float32, device=self.device)
        self.lse = torch.zeros((self.rows,), dtype=torch.float32, device=self.device)

    def load(self, q16, prefix_k16, prefix_v16, suffix_k16, suffix_v16):
        """q16[A, hq, d]; prefix_*[P, hkv, d]; suffix_*[A, S, hkv, d] (fp16, CUDA)."""
        self.q.copy_(q16)
        self.pk = encode_kv_head_major(self.k_fmt, prefix_k16, self.signs)
        self.pv = encode_kv_head_major(self.v_fmt, prefix_v16, self.signs)
        self.sk = encode_kv_head_major("f16", suffix_k16)
        self.sv = encode_kv_head_major("f16", suffix_v16)
        return self

    def build(self):
        """The step plan: the prefix part (every agent's rows in one pass over the shared
        prefix), the suffix part (each agent its own rows) and the combine; ``pre`` and
        ``suf`` keep the two parts' arguments."""
        self.pre = pre = attn_args(self.q, self.pk, self.pv, scale=self.scale, softcap=self.softcap,
                                   v_signs=self.signs, n_split=self.n_split_prefix, shared=True)
        self.suf = suf = attn_args(self.q, self.sk, self.sv, scale=self.scale, softcap=self.softcap,
                                   n_split=self.n_split_suffix)
        cap = attn_plan(pre)[0] + attn_plan(suf)[0]
        self.o_parts, self.lse_parts = _parts_buffers(cap, self.rows, self.d, self.device)
        self.plan = StepPlan([dict(device_parts=[pre, suf], tail=None, n_tiles=0,
                                   o_parts=self.o_parts, lse_parts=self.lse_parts,
                                   o=self.o, lse=self.lse)])
        return self

    def step(self, stream=None):
        self.plan.run(stream)

    def prefix_bytes(self) -> int:
        return self.pk.nbytes() + self.pv.nbytes()

    def suffix_bytes(self) -> int:
        return self.sk.nbytes() + self.sv.nbytes()
