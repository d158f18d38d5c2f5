"""The decode planner's logic with supplied measurements (no GPU): tier, window and ring
shape follow the policy oracle."""

import math

import pytest

from oracle import policy


@pytest.fixture(scope="module")
def autosize():
    from quantized_position_split_gb300 import autosize as a
    from quantized_position_split_gb300 import build
    build.build()
    return a


TIERS = [("f16", "f16"), ("q8_0", "q8_0"), ("q8_0", "tq3")]


def _per_token(hkv, d, kf, vf):
    row = {"f16": 2 * d, "q8_0": d + d // 16, "tq3": d // 4 + d // 8 + 2}
    return hkv * (row[kf] + row[vf])


@pytest.mark.parametrize("budget_frac,c_engage", [(1.5, 1.0), (0.7, 1.0), (0.7, 40.0), (0.2, 1.0), (0.05, 1.0)])
def test_plan_follows_the_policy(autosize, budget_frac, c_engage):
    layers, hq, hkv, d, n_kv = 48, 40, 8, 128, 65536
    f16_bytes = layers * n_kv * _per_token(hkv, d, "f16", "f16")
    budget = budget_frac * f16_bytes
    m = {"link_gbs": 211.0, "host_memcpy_gbs": 40.0, "c_engage_ms": c_engage, "attention_ms": 0.05, "vram_gbs": 6677.8}
    plan = autosize.plan_decode(layers=layers, batch=1, hq=hq, hkv=hkv, d=d, n_kv=n_kv, tiers=TIERS,
                                device_budget_bytes=budget, scale=0.088, measured=m, vram_gbs=6677.8)
    bw = 211.0  # the pinned link probe; the host CPU copy rate bounds nothing
    t_res = policy.t_resident_ms(0.0, f16_bytes, 6677.8)
    t_star = policy.t_star_bytes(t_res, c_engage, bw, 0.2)
    kv = [layers * n_kv * _per_token(hkv, d, kf, vf) for kf, vf in TIERS]
    tier = policy.choose_tier(kv, budget, t_star)
    assert plan["bw_eff_gbs"] == bw and math.isclose(plan["t_star_bytes"], t_star, rel_tol=1e-12)
    assert plan["tier"] == tier and (plan["k_fmt"], plan["v_fmt"]) == TIERS[tier]
    ptb = _per_token(hkv, d, *TIERS[tier])
    wc = min(n_kv, int(budget // (layers * ptb))) // 16 * 16
    assert plan["wc"] == wc and plan["tail_tokens"] == n_kv - wc
    if wc < n_kv:
        n, tiles, tb, tmax = policy.ring_plan(0.05, bw, max(budget - layers * wc * ptb, 1.0), (n_kv - wc) * ptb)
        assert plan["ring_slots"] == n
        assert plan["tile_tokens"] % 16 == 0 and 16 <= plan["tile_tokens"] <= max(16, tb // ptb)
    else:
        assert plan["ring_slots"] == 0
