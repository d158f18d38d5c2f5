"""Shared test helpers: workload assembly from the seeded generators and the parity
bar of the problem statement (per query row rel-L2 <= 1e-3 and max-abs <= 2e-3 on O,
|dLSE| <= 1e-4 on the same seeded inputs)."""

from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import pipeline

REL_L2 = 1e-3
MAX_ABS = 2e-3
LSE_ABS = 1e-4


def parity_report(o_gpu, lse_gpu, o_ref, lse_ref):
    o_gpu = np.asarray(o_gpu, dtype=np.float64).reshape(o_ref.shape)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64).reshape(lse_ref.shape)
    diff = o_gpu - o_ref
    den = np.linalg.norm(o_ref, axis=-1)
    rel = np.linalg.norm(diff, axis=-1) / np.where(den > 0, den, 1.0)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lse_gpu)), "empty / non-empty rows disagree"
    dl = np.abs(lse_gpu[fin] - lse_ref[fin])
    return dict(rel_l2=float(rel.max()), max_abs=float(np.abs(diff).max()),
                dlse=float(dl.max()) if dl.size else 0.0)


def assert_parity(o_gpu, lse_gpu, o_ref, lse_ref, tag=""):
    r = parity_report(o_gpu, lse_gpu, o_ref, lse_ref)
    assert r["rel_l2"] <= REL_L2 and r["max_abs"] <= MAX_ABS and r["dlse"] <= LSE_ABS, (tag, r)
    return r


def signs_for(cfg):
    """The workload's TurboQuant sign words, or its Rotation, for the library."""
    w1, w2, block = synth.rotation_words(cfg)
    if w2 is None and block == 0:
        return w1
    import quantized_position_split_gb300 as qps
    return qps.Rotation(w1, w2, block)


def oracle_signs(cfg):
    """The same rotation for the oracle."""
    from oracle import turboquant
    w1, w2, block = synth.rotation_words(cfg)
    if w2 is None and block == 0:
        return w1.numpy()
    return turboquant.Rotation(w1.numpy(), None if w2 is None else w2.numpy(), block or None)


def layer_inputs(cfg, layer, device):
    q = synth.query_f16(cfg, layer, device=device)
    k = synth.kv_f16(cfg, layer, "k", cfg.n_kv, device=device)
    v = synth.kv_f16(cfg, layer, "v", cfg.n_kv, device=device)
    return q, k, v


def oracle_layer(cfg, q, k, v):
    if cfg.mixed:
        return pipeline.mixed_layer_reference(q.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy(), cfg.wc,
                                              cfg.k_fmt, cfg.v_fmt, cfg.tk_fmt, cfg.tv_fmt, cfg.scale,
                                              cfg.softcap, oracle_signs(cfg))
    return pipeline.layer_reference(q.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy(),
                                    cfg.k_fmt, cfg.v_fmt, cfg.scale, cfg.softcap,
                                    oracle_signs(cfg))


def build_split_decoder(cfg, device="cuda", keep_inputs=(), **kw):
    """A PositionSplitDecoder for a "split" workload with all layers loaded.

    Returns (decoder, {layer: (q, k, v)} for the layers in keep_inputs (CPU tensors)).
    """
    from quantized_position_split_gb300.decode import PositionSplitDecoder

    dec = PositionSplitDecoder(layers=cfg.layers, batch=cfg.batch, hq=cfg.hq, hkv=cfg.hkv, d=cfg.d,
                               n_kv=cfg.n_kv, wc=cfg.wc, k_fmt=cfg.k_fmt, v_fmt=cfg.v_fmt,
                               scale=cfg.scale, softcap=cfg.softcap, signs=signs_for(cfg),
                               ring_slots=kw.pop("ring_slots", cfg.ring_slots),
                               tile_tokens=kw.pop("tile_tokens", cfg.tile_tokens), device=device,
                               tail_k_fmt=cfg.tail_k_fmt, tail_v_fmt=cfg.tail_v_fmt, **kw)
    kept = {}
    for layer in range(cfg.layers):
        q, k, v = layer_inputs(cfg, layer, device)
        dec.load_layer(layer, k, v, q[0:cfg.batch])
        if layer in keep_inputs:
            kept[layer] = (q.cpu(), k.cpu(), v.cpu())
        del k, v
    return dec.build(), kept


def fanout_inputs(cfg, device):
    q = synth.randn_f16((cfg.agents, cfg.hq, cfg.d), cfg.seed, cfg.name, "q", device=device)
    pk = synth.randn_f16((cfg.n_kv, cfg.hkv, cfg.d), cfg.seed, cfg.name, "prefix", "k", device=device)
    pv = synth.randn_f16((cfg.n_kv, cfg.hkv, cfg.d), cfg.seed, cfg.name, "prefix", "v", device=device)
    sk = synth.randn_f16((cfg.agents, cfg.suffix_len, cfg.hkv, cfg.d), cfg.seed, cfg.name, "suffix", "k",
                         device=device)
    sv = synth.randn_f16((cfg.agents, cfg.suffix_len, cfg.hkv, cfg.d), cfg.seed, cfg.name, "suffix", "v",
                         device=device)
    return q, pk, pv, sk, sv


def oracle_fanout(cfg, q, pk, pv, sk, sv):
    c = lambda t: t.cpu().numpy()  # noqa: E731
    return pipeline.fanout_reference(c(q), c(pk), c(pv), c(sk), c(sv), cfg.k_fmt, cfg.v_fmt,
                                     cfg.scale, cfg.softcap, oracle_signs(cfg))


def cuda_ok():
    return torch.cuda.is_available()
