"""The library's residency / ring sizing calls (host arithmetic) against the oracle."""

import numpy as np
import pytest

from oracle import policy


@pytest.fixture(scope="module")
def qps():
    import quantized_position_split_gb300 as q
    from quantized_position_split_gb300 import build
    build.build()
    return q


def test_plan_ring_matches_oracle(qps):
    rng = np.random.default_rng(3)
    for _ in range(500):
        c = float(rng.uniform(0.01, 20.0))
        bw = float(rng.uniform(1.0, 500.0))
        budget = float(rng.uniform(1e6, 5e10))
        tail = float(rng.choice([0.0, rng.uniform(1.0, 5e10)]))
        got = qps.plan_ring(c, bw, budget, tail)
        n, tiles, tb, tmax = policy.ring_plan(c, bw, budget, tail)
        assert (got["n_slots"], got["tiles_per_layer"], got["tile_bytes"], got["tile_bytes_max"]) == (n, tiles, tb, tmax)


def test_tail_band_and_tier_match_oracle(qps):
    rng = np.random.default_rng(4)
    for _ in range(500):
        t_res = float(rng.uniform(0.1, 200.0))
        c = float(rng.uniform(0.0, 5.0))
        bw = float(rng.uniform(1.0, 500.0))
        drop = float(rng.uniform(0.01, 0.9))
        t = qps.tail_band(t_res, c, bw, drop)
        assert t == policy.t_star_bytes(t_res, c, bw, drop)
        tiers = sorted(rng.uniform(1e6, 1e10, size=int(rng.integers(1, 5))).tolist(), reverse=True)
        budget = float(rng.uniform(0, 1e10))
        assert qps.choose_tier(tiers, budget, t) == policy.choose_tier(tiers, budget, t)


def test_policy_argument_errors(qps):
    from quantized_position_split_gb300 import _native as N
    for args in [(0.0, 1.0, 1.0, 1.0), (1.0, -1.0, 1.0, 1.0), (1.0, 1.0, 0.0, 1.0), (1.0, 1.0, 1.0, -1.0),
                 (float("nan"), 1.0, 1.0, 1.0)]:
        with pytest.raises(N.QpsError) as e:
            qps.plan_ring(*args)
        assert e.value.status == N.QPS_ERR_INVALID_ARG
    for args in [(0.0, 1.0, 1.0, 0.2), (1.0, -1.0, 1.0, 0.2), (1.0, 1.0, 0.0, 0.2), (1.0, 1.0, 1.0, 1.0)]:
        with pytest.raises(N.QpsError):
            qps.tail_band(*args)
    with pytest.raises(N.QpsError):
        qps.choose_tier([], 1.0, 0.0)
    with pytest.raises(N.QpsError):
        qps.choose_tier([1.0], 1.0, -1.0)


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5, 7])
def test_exact_boundaries_match_oracle(qps, k):
    """Budgets and tails that are exact multiples of the largest tile, and a tier whose
    bytes equal budget + T*: the floors, ceilings and the <= of both sides agree."""
    c, bw = 2.0, 200.0  # 320e6-byte tiles, exactly
    tmax = policy.ring_plan(c, bw, 1e9, 1.0)[3]
    for budget in (k * tmax, k * tmax * (1 - 1e-15), k * tmax * (1 + 1e-15)):
        for tail in (k * tmax, k * tmax + 1, k * tmax - 1):
            got = qps.plan_ring(c, bw, budget, tail)
            n, tiles, tb, tm = policy.ring_plan(c, bw, budget, tail)
            assert (got["n_slots"], got["tiles_per_layer"], got["tile_bytes"], got["tile_bytes_max"]) == \
                (n, tiles, tb, tm)
    t = qps.tail_band(50.0, 1.0, 200.0, 0.2)
    budget = 1e9
    tiers = [budget + t + 1.0, budget + t, budget + t - 1.0]
    assert qps.choose_tier(tiers, budget, t) == policy.choose_tier(tiers, budget, t) == 1
