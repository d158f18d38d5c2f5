"""Decode attention, position split and LSE combine (oracle, float64).

Sources:
  * "F5 M7 — Rolling KV: position-windowed KV residency", header status block: the KV
    cache is split by key position into a device window [0, wc) and a host tail
    [wc, n_kv), each attended separately and merged by an online-softmax combine.
  * Same page, section "Implementation decomposition, refined (S1 -> S2 -> S3)", item
    S2: each key tile yields its normalised output O_t and lse_t = m_t + log d_t; the
    merge is O = sum_t O_t exp(lse_t - M) / sum_t exp(lse_t - M) with M = max_t lse_t,
    done in f32 on the pages; a single tile reduces to plain attention.  The same item
    notes that the pages' streaming path only covered softcap == 0.
  * The problem statement: GQA-packed decode with an optional tanh logit softcap
    applied before the softmax.

Readings taken:
  * GQA mapping: query head h reads KV head h // (Hq / Hkv) (contiguous groups).
  * Logit: s = scale * <q, k>; with softcap c > 0, s <- c * tanh(s / c), before the
    max / exp; the LSE is taken over the capped logits.
  * LSE is the natural logarithm; O is normalised per part.
  * An empty part has lse = -inf and O = 0 and gets weight zero in the merge; if every
    part is empty the merged output is O = 0, lse = -inf.
"""

from __future__ import annotations

import math

import numpy as np


def logits(q: np.ndarray, k: np.ndarray, scale: float, softcap: float) -> np.ndarray:
    """s[r, j] = scale * <q_r, k_j>, then c * tanh(s / c) when softcap c > 0."""
    s = (np.asarray(q, dtype=np.float64) @ np.asarray(k, dtype=np.float64).T) * scale
    if softcap > 0:
        s = softcap * np.tanh(s / softcap)
    return s


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, softcap: float = 0.0):
    """Softmax attention of rows ``q[R, D]`` over ``k[n, D]``, ``v[n, Dv]``.

    Returns ``(O [R, Dv], lse [R])`` with O normalised.  n == 0 gives O = 0, lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    r = q.shape[0]
    n = k.shape[0]
    dv = v.shape[-1]
    if n == 0:
        return np.zeros((r, dv)), np.full(r, -np.inf)
    s = logits(q, k, scale, softcap)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ np.asarray(v, dtype=np.float64)) / l
    lse = (m + np.log(l))[:, 0]
    return o, lse


def gqa_decode(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
               softcap: float = 0.0, begin: int = 0, end=None):
    """Decode attention of ``q[B, Hq, D]`` over token-major ``k, v[n, Hkv, D]``.

    All B query rows of a head read the same KV (B = 1 for a single sequence; B > 1
    for agents sharing one prefix).  Only positions [begin, end) are attended.
    Returns ``(O [B, Hq, D], lse [B, Hq])``.
    """
    q = np.asarray(q, dtype=np.float64)
    b, hq, d = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    n = k.shape[0]
    end = n if end is None else end
    o = np.zeros((b, hq, v.shape[-1]))
    lse = np.zeros((b, hq))
    for h in range(hq):
        kv = h // g
        oh, lh = attend(q[:, h, :], k[begin:end, kv, :], v[begin:end, kv, :], scale, softcap)
        o[:, h, :] = oh
        lse[:, h] = lh
    return o, lse


def multi_query_decode(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                       softcap: float = 0.0, begin: int = 0, end=None, q_pos=None):
    """Attention of ``n_q`` query tokens of one sequence, ``q[n_q, Hq, D]``, over
    token-major ``k, v[n, Hkv, D]`` (positions [begin, end)).

    The verify batch of "F5 M6 — PolyKV (shared compressed KV pool)", section "S2
    perf-path — turbo-MMA verify kernel + scalar-K/turbo-V fused decode" (n_q > 1 query
    tokens checked in one pass over the cache).  With ``q_pos`` given, query token i
    sits at position ``q_pos + i`` of the same index space and sees only the positions
    p <= q_pos + i (the cache up to and including itself); without it every query sees
    all of [begin, end).  Returns ``(O [n_q, Hq, D], lse [n_q, Hq])``; a query that sees
    no position gets O = 0, lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    n_q = q.shape[0]
    end = k.shape[0] if end is None else end
    o = np.zeros((n_q,) + q.shape[1:2] + (v.shape[-1],))
    lse = np.zeros(q.shape[:2])
    for i in range(n_q):
        e = end if q_pos is None else min(end, max(begin, q_pos + i + 1))
        oi, li = gqa_decode(q[i:i + 1], k, v, scale, softcap, begin, e)
        o[i], lse[i] = oi[0], li[0]
    return o, lse


def lse_combine(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge normalised partial outputs by their log-sum-exp.

    ``o_parts[P, ..., D]``, ``lse_parts[P, ...]`` -> ``(O [..., D], lse [...])``:
    M = max_t lse_t, w_t = exp(lse_t - M), O = sum_t w_t O_t / sum_t w_t,
    lse = M + log sum_t w_t; parts with lse = -inf have weight 0.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.max(lse_parts, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - m_safe[None]), 0.0)
    den = w.sum(axis=0)
    num = np.einsum("p...,p...d->...d", w, o_parts)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(finite[..., None], num / np.where(den > 0, den, 1.0)[..., None], 0.0)
        lse = np.where(finite, m_safe + np.log(np.where(den > 0, den, 1.0)), -np.inf)
    return o, lse


def split_decode(q, k, v, wc: int, scale: float, softcap: float = 0.0, tail_tiles=None):
    """Window [0, wc) and tail [wc, n) attended separately, then merged.

    ``tail_tiles`` (optional) is a list of (begin, end) ranges tiling the tail; each
    tile becomes its own part, as the streamed tail does.
    """
    n = k.shape[0]
    parts = [gqa_decode(q, k, v, scale, softcap, 0, wc)]
    if tail_tiles is None:
        tail_tiles = [(wc, n)]
    for a, b in tail_tiles:
        parts.append(gqa_decode(q, k, v, scale, softcap, a, b))
    o_parts = np.stack([p[0] for p in parts])
    lse_parts = np.stack([p[1] for p in parts])
    return lse_combine(o_parts, lse_parts)


def attend_loops(q, k, v, scale: float, softcap: float = 0.0):
    """The same as ``attend`` written as explicit Python loops (tiny inputs only)."""
    q = [[float(x) for x in row] for row in np.asarray(q)]
    k = [[float(x) for x in row] for row in np.asarray(k)]
    v = [[float(x) for x in row] for row in np.asarray(v)]
    dv = len(v[0]) if v else 0
    outs, lses = [], []
    for qr in q:
        s = []
        for kr in k:
            acc = 0.0
            for a, b in zip(qr, kr):
                acc += a * b
            acc *= scale
            if softcap > 0:
                acc = softcap * math.tanh(acc / softcap)
            s.append(acc)
        if not s:
            outs.append([0.0] * dv)
            lses.append(-math.inf)
            continue
        m = max(s)
        e = [math.exp(x - m) for x in s]
        den = sum(e)
        o = [0.0] * dv
        for w, vr in zip(e, v):
            for i in range(dv):
                o[i] += w * vr[i]
        outs.append([x / den for x in o])
        lses.append(m + math.log(den))
    return np.array(outs), np.array(lses)
