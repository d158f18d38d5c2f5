"""Pins of the Lloyd-Max codebook against J. Max's published table and the
optimality conditions."""

import math

import numpy as np
from scipy import integrate
from scipy.stats import norm

from oracle import turboquant as tq
from tests.conftest import golden_rows


def _max_table():
    rows = golden_rows("max1960_gaussian_8level.txt")
    out = {"output": [], "threshold": [], "mse": []}
    for kind, val in rows:
        out[kind].append(float(val))
    return out


def test_lloyd_matches_max_1960_table():
    tab = _max_table()
    c, t = tq.lloyd_max_gaussian(8)
    pos = c[4:]
    for got, want in zip(pos, tab["output"]):
        assert abs(got - want) <= 6e-4 * max(1.0, abs(want)), (got, want)
    for got, want in zip(t[3:], tab["threshold"]):
        assert abs(got - want) <= 6e-4 * max(1.0, abs(want)), (got, want)
    mse = tq.gaussian_mse(c, t)
    assert abs(mse - tab["mse"][0]) < 1e-5


def test_centroid_condition_by_quadrature():
    """Each level is the mean of N(0,1) over its cell (scipy quadrature, not the
    closed form the solver uses)."""
    c, t = tq.lloyd_max_gaussian(8)
    edges = np.concatenate([[-np.inf], t, [np.inf]])
    for k in range(8):
        a, b = edges[k], edges[k + 1]
        num, _ = integrate.quad(lambda x: x * norm.pdf(x), a, b, epsabs=1e-14, epsrel=1e-13)
        den = norm.cdf(b) - norm.cdf(a)
        assert abs(num / den - c[k]) < 1e-9


def test_midpoint_condition_and_symmetry():
    c, t = tq.lloyd_max_gaussian(8)
    assert np.allclose(t, 0.5 * (c[:-1] + c[1:]), atol=0, rtol=0)
    assert np.allclose(c, -c[::-1], atol=1e-12)
    assert np.all(np.diff(c) > 0)


def test_build_codebook_is_fp16_exact_and_near_optimal():
    levels, thr = tq.codebook()
    c, _ = tq.lloyd_max_gaussian(8)
    assert levels.dtype == np.float32 and thr.dtype == np.float32
    # levels exactly representable in fp16, within one fp16 rounding of Lloyd-Max
    assert np.array_equal(levels.astype(np.float16).astype(np.float32), levels)
    assert np.all(np.abs(levels - c) <= np.abs(c) * 2.0 ** -11)
    # exactly symmetric; thresholds exactly the midpoints (checked in float64)
    assert np.array_equal(levels, -levels[::-1])
    assert np.array_equal(thr.astype(np.float64),
                          0.5 * (levels[:-1].astype(np.float64) + levels[1:].astype(np.float64)))
    # the distortion moves by far less than the table's precision
    assert abs(tq.gaussian_mse(levels, thr) - tq.gaussian_mse(c, 0.5 * (c[:-1] + c[1:]))) < 1e-6


def test_monte_carlo_distortion_by_brute_force_nearest():
    levels, _ = tq.codebook()
    rng = np.random.default_rng(3)
    x = rng.standard_normal(400000)
    nearest = levels.astype(np.float64)[np.argmin(np.abs(x[:, None] - levels[None, :]), axis=1)]
    mse = float(np.mean((x - nearest) ** 2))
    assert abs(mse - _max_table()["mse"][0]) < 4e-4


def test_threshold_count_rule_equals_nearest_level():
    levels, thr = tq.codebook()
    rng = np.random.default_rng(4)
    z = rng.standard_normal(50000).astype(np.float32) * 1.5
    k = np.zeros(z.shape, dtype=np.int64)
    for t in thr:
        k += (z >= t)
    nearest = np.argmin(np.abs(z[:, None].astype(np.float64) - levels[None, :].astype(np.float64)), axis=1)
    assert np.array_equal(k, nearest)
    assert math.isclose(float(thr[3]), 0.0, abs_tol=0.0)


def test_every_oracle_function_is_documented_and_every_module_cites_its_pages():
    import inspect

    from oracle import attention, pipeline, policy, q8_0
    for m in (attention, q8_0, tq, pipeline, policy):
        assert '"F5 M' in m.__doc__ or '"T*-aware' in m.__doc__ or '"Rolling-KV' in m.__doc__, m.__name__
        for name, f in vars(m).items():
            if inspect.isfunction(f) and f.__module__ == m.__name__:
                assert f.__doc__, f"{m.__name__}.{name}"
