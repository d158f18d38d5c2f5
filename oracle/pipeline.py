"""Whole-layer expected outputs from fp16 inputs (oracle).

The oracle encodes the fp16 K / V itself with its own encoders, dequantises them to
float64, and computes plain (unsplit) decode attention over every position: by the
combine identity of "F5 M7 — Rolling KV: position-windowed KV residency" (section
"Implementation decomposition, refined (S1 -> S2 -> S3)", item S2) this is what the
position-split path must reproduce for every window length.

The shared-prefix workload follows "F5 M6 — PolyKV (shared compressed KV pool)",
section "S1 — SharedKVPool": one compressed prefix read by every agent, plus a
private suffix per agent; agent b attends prefix + suffix_b.
"""

from __future__ import annotations

import numpy as np

from . import attention, q8_0, turboquant


def encode(fmt: str, x16: np.ndarray, sign_words=None):
    """Stored planes of ``x16[..., D]`` in format ``fmt`` (tuple of arrays)."""
    x16 = np.asarray(x16, dtype=np.float16)
    if fmt == "f16":
        return (x16,)
    if fmt == "q8_0":
        return q8_0.encode(x16)
    if fmt == "tq3":
        return turboquant.encode(x16, sign_words)
    if fmt in ("tq2", "tq4"):
        planes, norms = turboquant.encode_tier(x16, sign_words, int(fmt[2]))
        return planes + (norms,)
    raise ValueError(fmt)


def dequant(fmt: str, x16: np.ndarray, sign_words=None) -> np.ndarray:
    """What the attention reads for ``x16`` stored in ``fmt``, in float64."""
    x16 = np.asarray(x16, dtype=np.float16)
    d = x16.shape[-1]
    if fmt == "f16":
        return x16.astype(np.float64)
    if fmt == "q8_0":
        return q8_0.decode(*q8_0.encode(x16))
    if fmt == "tq3":
        lo2, hi1, n = turboquant.encode(x16, sign_words)
        return turboquant.decode(lo2, hi1, n, sign_words, d)
    if fmt in ("tq2", "tq4"):
        bits = int(fmt[2])
        planes, n = turboquant.encode_tier(x16, sign_words, bits)
        return turboquant.decode_tier(planes, n, sign_words, d, bits)
    raise ValueError(fmt)


def layer_reference(q16, k16, v16, k_fmt: str, v_fmt: str, scale: float, softcap: float,
                    sign_words=None):
    """Expected (O [B, Hq, D], lse [B, Hq]) of one layer over all positions.

    ``q16[B, Hq, D]``, ``k16, v16[n, Hkv, D]`` are the fp16 inputs; K and V are read
    through their stored formats.
    """
    kh = dequant(k_fmt, k16, sign_words)
    vh = dequant(v_fmt, v16, sign_words)
    return attention.gqa_decode(np.asarray(q16, dtype=np.float64), kh, vh, scale, softcap)


def mixed_layer_reference(q16, k16, v16, wc: int, k_fmt: str, v_fmt: str, tail_k_fmt: str,
                          tail_v_fmt: str, scale: float, softcap: float, sign_words=None):
    """Expected outputs of one layer whose tail carries other storage formats.

    "F5 M7 — Rolling KV: position-windowed KV residency", section "2026-07-12 — #582-P2
    SHIPPED: position-axis mixed KV (compressed tail, -ctkt/-ctvt)": the positions
    [0, wc) keep the window's K / V formats, the positions [wc, n) are stored in the
    tail's (more compressed) formats, and each part is read at its own format.  The
    expected output is plain attention over the concatenation of the two dequantised
    ranges; with the tail formats equal to the window's it is ``layer_reference``.
    """
    kh = np.concatenate([dequant(k_fmt, k16[:wc], sign_words), dequant(tail_k_fmt, k16[wc:], sign_words)], axis=0)
    vh = np.concatenate([dequant(v_fmt, v16[:wc], sign_words), dequant(tail_v_fmt, v16[wc:], sign_words)], axis=0)
    return attention.gqa_decode(np.asarray(q16, dtype=np.float64), kh, vh, scale, softcap)


def fanout_reference(q16, prefix_k16, prefix_v16, suffix_k16, suffix_v16,
                     k_fmt: str, v_fmt: str, scale: float, softcap: float = 0.0,
                     sign_words=None):
    """Expected outputs of the shared-prefix workload.

    ``q16[A, Hq, D]`` (one query token per agent), ``prefix_*[P, Hkv, D]`` stored in
    (k_fmt, v_fmt), ``suffix_*[A, S, Hkv, D]`` fp16.  Agent a attends prefix + suffix_a.
    """
    kp = dequant(k_fmt, prefix_k16, sign_words)
    vp = dequant(v_fmt, prefix_v16, sign_words)
    q = np.asarray(q16, dtype=np.float64)
    a_n = q.shape[0]
    o = np.zeros(q.shape)
    lse = np.zeros(q.shape[:2])
    for a in range(a_n):
        k = np.concatenate([kp, np.asarray(suffix_k16[a], dtype=np.float64)], axis=0)
        v = np.concatenate([vp, np.asarray(suffix_v16[a], dtype=np.float64)], axis=0)
        oa, la = attention.gqa_decode(q[a:a + 1], k, v, scale, softcap)
        o[a] = oa[0]
        lse[a] = la[0]
    return o, lse
