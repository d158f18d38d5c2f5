"""Assembly of a whole position-split decode step from per-layer fp16 K / V caches.

Each layer's cache is encoded on the GPU by the library's encoders, its window
[0, wc) stays in device memory, and its tail [wc, n_kv) is copied once to pinned host
memory, token-major, so that a tile of consecutive positions is one contiguous range
per plane ("Rolling-KV: step/graph-level tail prefetch (design)", section "The fix: a
persistent, step-spanning tail-prefetch ring"; "F5 M7 — Rolling KV: position-windowed
KV residency", header status block).  A step is one ``qps_decode_step`` call: per
layer, the window part, the layer's ring tiles, and the LSE combine.

The shared-prefix batch ("F5 M6 — PolyKV (shared compressed KV pool)", section "S1 —
SharedKVPool") is assembled by ``FanoutDecoder``: one compressed prefix read by every
agent in one pass, plus one private fp16 suffix per agent, merged per agent.
"""

from __future__ import annotations

from typing import List, Optional

import torch

from . import KV, Ring, StepPlan, attn_args, attn_plan, encode_kv, tile_desc


def _parts_buffers(capacity: int, rows: int, d: int, device):
    return (torch.empty((capacity, rows, d), dtype=torch.float32, device=device),
            torch.empty((capacity, rows), dtype=torch.float32, device=device))


class PositionSplitDecoder:
    """Decode attention of ``layers`` layers over a KV cache split at ``wc``."""

    def __init__(self, *, layers: int, batch: int, hq: int, hkv: int, d: int, n_kv: int, wc: int,
                 k_fmt: str, v_fmt: str, scale: float, softcap: float = 0.0, signs=None,
                 ring_slots: int = 3, tile_tokens: int = 8192, n_split_window: int = 0,
                 n_split_tail: int = 0, device=None):
        if not 0 <= wc <= n_kv:
            raise ValueError("need 0 <= wc <= n_kv")
        self.layers, self.batch, self.hq, self.hkv, self.d = layers, batch, hq, hkv, d
        self.n_kv, self.wc = n_kv, wc
        self.k_fmt, self.v_fmt = k_fmt, v_fmt
        self.scale, self.softcap, self.signs = scale, softcap, signs
        self.ring_slots, self.tile_tokens = ring_slots, tile_tokens
        self.n_split_window, self.n_split_tail = n_split_window, n_split_tail
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.rows = batch * hq
        self.q = torch.zeros((layers, batch, hq, d), dtype=torch.float16, device=self.device)
        self.o = torch.zeros((layers, self.rows, d), dtype=torch.float32, device=self.device)
        self.lse = torch.zeros((layers, self.rows), dtype=torch.float32, device=self.device)
        self.window: List[Optional[tuple]] = [None] * layers  # (K, V) on device
        self.tail: List[Optional[tuple]] = [None] * layers  # (K, V) pinned host
        self.ring: Optional[Ring] = None
        self.plan: Optional[StepPlan] = None
        self.window_plan: Optional[StepPlan] = None

    @property
    def tail_len(self) -> int:
        return self.n_kv - self.wc

    def tile_ranges(self):
        t = self.tile_tokens
        return [(a, min(a + t, self.tail_len)) for a in range(0, self.tail_len, t)]

    def load_layer(self, layer: int, k16: torch.Tensor, v16: torch.Tensor, q16: Optional[torch.Tensor] = None):
        """Encode one layer's fp16 ``k16, v16[n_kv, hkv, d]`` (CUDA) and place it."""
        k = encode_kv(self.k_fmt, k16, self.signs)
        v = encode_kv(self.v_fmt, v16, self.signs)
        torch.cuda.current_stream().synchronize()
        kw, vw = k.token_slice(0, self.wc), v.token_slice(0, self.wc)
        # the window keeps its own storage so the full-length encode can be freed
        kw = KV(kw.fmt, tuple(p.clone() for p in kw.planes), kw.tokens, kw.hkv, kw.d, kw.tok_stride)
        vw = KV(vw.fmt, tuple(p.clone() for p in vw.planes), vw.tokens, vw.hkv, vw.d, vw.tok_stride)
        self.window[layer] = (kw, vw)
        if self.tail_len > 0:
            self.tail[layer] = (k.token_slice(self.wc, self.n_kv).pinned_copy(),
                                v.token_slice(self.wc, self.n_kv).pinned_copy())
        if q16 is not None:
            self.q[layer].copy_(q16)

    def _args(self, layer, k: KV, v: KV, n_split: int):
        return attn_args(self.q[layer], k, v, scale=self.scale, softcap=self.softcap,
                         v_signs=self.signs, n_split=n_split)

    def build(self):
        """Create the ring, the flat (layer, tile) schedule and the step plans."""
        ranges = self.tile_ranges()
        tiles = []
        slot_bytes = 0
        if self.tail_len > 0:
            for layer in range(self.layers):
                kt, vt = self.tail[layer]
                for a, b in ranges:
                    td = tile_desc(kt, vt, a, b)
                    tiles.append(td)
                    need = sum((x + 255) // 256 * 256 for x in list(td.bytes_k) + list(td.bytes_v))
                    slot_bytes = max(slot_bytes, need)
            self.ring = Ring(self.ring_slots, slot_bytes, self.device.index)
        layers, wlayers = [], []
        self._keep = []
        self.window_args = []
        for layer in range(self.layers):
            kw, vw = self.window[layer]
            wargs = self._args(layer, kw, vw, self.n_split_window)
            self.window_args.append(wargs)
            n_w, _ = attn_plan(wargs)
            cap = n_w
            tail_tpl = None
            if self.tail_len > 0:
                kt, vt = self.tail[layer]
                # a template: the ring replaces the data pointers with its slot's planes
                tail_tpl = self._args(layer, kt, vt, self.n_split_tail)
                for a, b in ranges:
                    probe = self._args(layer, kt.token_slice(a, b), vt.token_slice(a, b), self.n_split_tail)
                    cap += attn_plan(probe)[0]
            o_parts, lse_parts = _parts_buffers(cap, self.rows, self.d, self.device)
            self._keep += [o_parts, lse_parts]
            layers.append(dict(device_parts=[wargs], tail=tail_tpl,
                               n_tiles=len(ranges) if self.tail_len > 0 else 0,
                               o_parts=o_parts, lse_parts=lse_parts, o=self.o[layer], lse=self.lse[layer]))
            wlayers.append(dict(device_parts=[wargs], tail=None, n_tiles=0,
                                o_parts=o_parts, lse_parts=lse_parts, o=self.o[layer], lse=self.lse[layer]))
        self.plan = StepPlan(layers, tiles, self.ring)
        self.window_plan = StepPlan(wlayers)
        self.n_tiles = len(tiles)
        return self

    def step(self, stream=None):
        self.plan.run(stream)

    def window_step(self, stream=None):
        """The same step with the ring and the tail omitted (window parts + combines)."""
        self.window_plan.run(stream)

    # algorithmic bytes: every stored plane the step must read once
    def window_bytes(self) -> int:
        return sum(kv.nbytes() for w in self.window for kv in w)

    def tail_bytes(self) -> int:
        return sum(kv.nbytes() for t in self.tail if t is not None for kv in t)

    def close(self):
        if self.ring is not None:
            self.ring.close()
            self.ring = None


class FanoutDecoder:
    """One compressed prefix shared by ``agents`` query rows sets, plus private fp16
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
        self.pk = encode_kv(self.k_fmt, prefix_k16, self.signs)
        self.pv = encode_kv(self.v_fmt, prefix_v16, self.signs)
        self.sk = encode_kv("f16", suffix_k16)
        self.sv = encode_kv("f16", suffix_v16)
        return self

    def build(self):
        pre = attn_args(self.q, self.pk, self.pv, scale=self.scale, softcap=self.softcap,
                        v_signs=self.signs, n_split=self.n_split_prefix, shared=True)
        suf = attn_args(self.q, self.sk, self.sv, scale=self.scale, softcap=self.softcap,
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
