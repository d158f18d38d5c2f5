"""Measured decode planning on the GPU: the probes return sane figures and a decoder
built from the plan (tier, window, ring shape) matches the oracle."""

import numpy as np
import pytest
import torch

import synth
from tests import helpers
from tests.helpers import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qps():
    import quantized_position_split_gb300 as q
    from quantized_position_split_gb300 import build
    build.build()
    return q


def test_probes_are_sane(qps):
    from quantized_position_split_gb300 import autosize
    dev = torch.device("cuda", 0)
    link, host = autosize.measure_link(dev, nbytes=64 << 20)
    assert 1.0 < link < 2000.0 and host > 0.1
    words = synth.sign_bits(128, 42)
    ms = autosize.attention_ms("q8_0", "tq3", batch=1, hq=8, hkv=2, d=128, n_kv=4096, scale=0.088,
                               signs=words, device=dev, reps=5)
    assert 0.0 < ms < 50.0
    c = autosize.c_engage_ms("q8_0", "q8_0", batch=1, hq=8, hkv=2, d=128, n_kv=4096, scale=0.088,
                             device=dev, reps=5)
    assert 0.0 <= c < 50.0


def test_planned_decoder_matches_oracle(qps):
    from quantized_position_split_gb300 import autosize
    from quantized_position_split_gb300.decode import PositionSplitDecoder
    cfg = synth.parity_scaled(synth.by_name("qwen14b_f16"), layers=2)
    tiers = [("f16", "f16"), ("q8_0", "q8_0"), ("q8_0", "tq3")]
    per_tok_f16 = cfg.hkv * 2 * (2 * cfg.d)
    budget = 0.6 * cfg.layers * cfg.n_kv * per_tok_f16
    signs = helpers.signs_for(cfg)
    plan = autosize.plan_decode(layers=cfg.layers, batch=cfg.batch, hq=cfg.hq, hkv=cfg.hkv, d=cfg.d,
                                n_kv=cfg.n_kv, tiers=tiers, device_budget_bytes=budget, scale=cfg.scale,
                                signs=signs, measured={"c_engage_ms": 0.0})
    assert 0 <= plan["wc"] <= cfg.n_kv and plan["wc"] % 16 == 0
    assert plan["tail_tokens"] > 0 and 2 <= plan["ring_slots"] <= 4 and plan["tile_tokens"] >= 16
    run = cfg.replace(k_fmt=plan["k_fmt"], v_fmt=plan["v_fmt"], wc=plan["wc"], ring_slots=plan["ring_slots"],
                      tile_tokens=min(plan["tile_tokens"], 1024))
    dec, kept = helpers.build_split_decoder(run, keep_inputs=range(run.layers))
    dec.step()
    torch.cuda.synchronize()
    for layer, (q, k, v) in kept.items():
        ro, rl = helpers.oracle_layer(run, q, k, v)
        assert_parity(dec.o[layer].cpu().numpy(), dec.lse[layer].cpu().numpy(), ro.reshape(-1, run.d),
                      rl.reshape(-1), (plan["k_fmt"], plan["v_fmt"], plan["wc"], layer))
    dec.ring.sync()
    dec.close()
