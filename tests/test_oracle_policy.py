"""Pins of the residency / ring sizing oracle against the pages' anchor, invariants of
the formulas and hand-checked boundaries."""

import math
import os

import pytest

from oracle import policy

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tstar_anchor.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_t_star_anchor_rtx3090():
    g = _golden()
    t = policy.t_star_bytes(g["t_resident_ms"], g["c_engage_ms"], g["bw_eff_gbs"], g["target_drop"])
    assert g["t_star_mib_min"] <= t / 2**20 <= g["t_star_mib_max"]


@pytest.mark.parametrize("t_res,c,bw", [(23.6, 1.4, 6.5), (100.0, 2.0, 211.0), (5.0, 0.1, 50.0)])
def test_drop_at_t_star_is_the_target(t_res, c, bw):
    """The defining property: streaming exactly T* costs exactly the target drop."""
    t = policy.t_star_bytes(t_res, c, bw, 0.2)
    assert t > 0
    assert math.isclose(policy.tail_drop(c, t, bw, t_res), 0.2, rel_tol=1e-12)
    assert policy.tail_drop(c, 2 * t, bw, t_res) > 0.2 > policy.tail_drop(c, t / 2, bw, t_res)


def test_short_context_never_spills():
    """A small resident time cannot absorb the engagement cost: T* = 0 (quantise)."""
    assert policy.t_star_bytes(5.0, 1.4, 211.0, 0.2) == 0.0
    assert policy.t_star_bytes(6.99, 1.4, 211.0, 0.2) == 0.0  # 0.2 * 6.99 < 1.4: none


def test_t_resident_is_bytes_over_bandwidth():
    assert math.isclose(policy.t_resident_ms(20e9, 10e9, 6000.0), 5.0, rel_tol=1e-12)


def test_choose_tier():
    tiers = [100, 60, 35]  # f16, q8_0, a more compressed tier
    assert policy.choose_tier(tiers, 120, 0) == 0  # everything fits: f16
    assert policy.choose_tier(tiers, 90, 10) == 0  # f16 spills 10 <= T*: keep f16 and spill
    assert policy.choose_tier(tiers, 90, 9) == 1   # f16 spill past T*: q8_0 fits
    assert policy.choose_tier(tiers, 30, 4) == 2   # 35 <= 34? no; nothing fits: the floor
    assert policy.choose_tier(tiers, 30, 5) == 2


def test_ring_plan_boundaries():
    # 2 ms per layer at 200 GB/s with the 0.8 safety: 320 MB tiles
    n, tiles, tb, tmax = policy.ring_plan(2.0, 200.0, 1e9, 1000e6)
    assert math.isclose(tmax, 320e6, rel_tol=1e-12)
    assert n == 3 and tiles == 4 and tb == 250e6
    assert tiles * tb >= 1000e6 and (tiles - 1) * tmax < 1000e6 and tb <= tmax
    assert policy.ring_plan(2.0, 200.0, 100e6, 1e6)[0] == 2   # budget below two tiles: 2
    assert policy.ring_plan(2.0, 200.0, 10e9, 1e6)[0] == 4    # large budget: at most 4
    assert policy.ring_plan(2.0, 200.0, 1e9, 0)[1:3] == (0, 0)  # no tail: no tiles
    assert policy.ring_plan(2.0, 200.0, 1e9, 320e6)[1] == 1    # exactly one tile


@pytest.mark.parametrize("tail", [1000e6 + 1, 999_999_999.0, 7.0, 641e6, 123_456_789.0])
def test_ring_tiles_cover_a_tail_that_does_not_divide(tail):
    """Brute force over tile counts: the plan takes the fewest equal tiles no larger
    than the maximum, and those tiles (whole bytes) cover the whole tail."""
    n, tiles, tb, tmax = policy.ring_plan(2.0, 200.0, 1e9, tail)
    fewest = next(t for t in range(1, 10 ** 6) if tail / t <= tmax)
    assert tiles == fewest
    assert tb == int(tb) and tiles * tb >= tail and (tiles - 1) * tb < tail
    assert tb <= tmax + 1
