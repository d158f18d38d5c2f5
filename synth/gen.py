"""Seeded random draws (torch Philox generators keyed by a hash of string tags)."""

from __future__ import annotations

import hashlib
from typing import Optional, Sequence

import torch


def seed_for(base_seed: int, *tags) -> int:
    """A 63-bit generator seed derived from a base seed and any number of tags."""
    h = hashlib.blake2b(digest_size=8)
    h.update(str(int(base_seed)).encode())
    for t in tags:
        h.update(b"\x00")
        h.update(str(t).encode())
    return int.from_bytes(h.digest(), "little") & ((1 << 63) - 1)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def outlier_channels(base_seed: int, layer: int, hkv: int, d: int, count: int) -> torch.Tensor:
    """``count`` distinct channel indices per KV head, shape [hkv, count] (int64, CPU)."""
    out = torch.empty((hkv, count), dtype=torch.int64)
    for h in range(hkv):
        g = _gen("cpu", seed_for(base_seed, "outliers", layer, h))
        out[h] = torch.randperm(d, generator=g)[:count]
    return out


def randn_f16(shape: Sequence[int], base_seed: int, *tags, device="cpu",
              channel_scale: Optional[torch.Tensor] = None) -> torch.Tensor:
    """N(0,1) float32 draws rounded to fp16.

    ``channel_scale`` (float32, broadcastable to ``shape``) multiplies the draws before
    the rounding; it is how outlier channels are planted.
    """
    g = _gen(device, seed_for(base_seed, *tags))
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if channel_scale is not None:
        x = x * channel_scale.to(device=device, dtype=torch.float32)
    return x.to(torch.float16)


def kv_f16(cfg, layer: int, which: str, tokens: int, token_offset_tag: str = "",
           device="cpu") -> torch.Tensor:
    """K or V of one layer as fp16 [tokens, hkv, d] (token-major).

    K carries ``cfg.k_outliers`` outlier channels per KV head (scaled by
    ``cfg.outlier_scale``); V never does.
    """
    scale = None
    if which == "k" and cfg.k_outliers > 0:
        ch = outlier_channels(cfg.seed, layer, cfg.hkv, cfg.d, cfg.k_outliers)
        scale = torch.ones((cfg.hkv, cfg.d), dtype=torch.float32)
        for h in range(cfg.hkv):
            scale[h, ch[h]] = cfg.outlier_scale
        scale = scale.unsqueeze(0)
    return randn_f16((tokens, cfg.hkv, cfg.d), cfg.seed, cfg.name, "kv", which, layer,
                     token_offset_tag, device=device, channel_scale=scale)


def query_f16(cfg, layer: int, device="cpu", tag: str = "") -> torch.Tensor:
    """The decode query of one layer, fp16 [batch, hq, d]."""
    return randn_f16((cfg.batch, cfg.hq, cfg.d), cfg.seed, cfg.name, "q", layer, tag,
                     device=device)


def rotation_words(cfg):
    """A workload's TurboQuant rotation inputs: (sign words s1, sign words s2 or None,
    Hadamard block width, 0 = head_dim)."""
    w2 = None if cfg.sign_seed2 is None else sign_bits(cfg.d, cfg.sign_seed2)
    return sign_bits(cfg.d, cfg.sign_seed), w2, cfg.rot_block


def sign_bits(d: int, seed: int = 42) -> torch.Tensor:
    """The seeded sign diagonal as d/32 uint32 words (int64 tensor holding the words).

    Bit i of word i // 32 set means s_i = -1.
    """
    if d % 32:
        raise ValueError("d must be a multiple of 32")
    g = _gen("cpu", seed_for(seed, "tq-signs", d))
    bits = torch.randint(0, 2, (d,), generator=g, dtype=torch.int64)
    words = torch.zeros(d // 32, dtype=torch.int64)
    for i in range(d):
        if bits[i]:
            words[i // 32] |= 1 << (i % 32)
    return words
