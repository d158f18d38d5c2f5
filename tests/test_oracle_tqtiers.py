"""Pins of the 2- and 4-bit TurboQuant tiers: their codebooks against J. Max's table
and the optimality conditions, the plane layouts bit by bit, nearest-level codes and
the distortion ladder."""

import numpy as np
import pytest
from scipy import integrate
from scipy.stats import norm

from oracle import turboquant as tq
from tests.conftest import golden_rows

TABLES = {4: "max1960_gaussian_4level.txt", 16: "max1960_gaussian_16level.txt"}


def _table(levels):
    out = {"output": [], "threshold": [], "mse": []}
    for kind, val in golden_rows(TABLES[levels]):
        out[kind].append(float(val))
    return out


@pytest.mark.parametrize("levels", [4, 16])
def test_lloyd_matches_max_1960_table(levels):
    tab = _table(levels)
    c, t = tq.lloyd_max_gaussian(levels)
    h = levels // 2
    for got, want in zip(c[h:], tab["output"]):
        assert abs(got - want) <= 6e-4 * max(1.0, abs(want)), (got, want)
    for got, want in zip(t[h - 1:], tab["threshold"]):
        assert abs(got - want) <= 6e-4 * max(1.0, abs(want)), (got, want)
    assert abs(tq.gaussian_mse(c, t) - tab["mse"][0]) < 2e-5


@pytest.mark.parametrize("levels", [4, 16])
def test_centroid_condition_by_quadrature(levels):
    c, t = tq.lloyd_max_gaussian(levels)
    edges = np.concatenate([[-np.inf], t, [np.inf]])
    for k in range(levels):
        a, b = edges[k], edges[k + 1]
        num, _ = integrate.quad(lambda x: x * norm.pdf(x), a, b, epsabs=1e-14, epsrel=1e-13)
        assert abs(num / (norm.cdf(b) - norm.cdf(a)) - c[k]) < 1e-9


@pytest.mark.parametrize("levels", [4, 16])
def test_build_codebook_fp16_exact_symmetric_midpoints(levels):
    lv, thr = tq.codebook(levels)
    c, _ = tq.lloyd_max_gaussian(levels)
    assert np.array_equal(lv.astype(np.float16).astype(np.float32), lv)
    assert np.all(np.abs(lv - c) <= np.abs(c) * 2.0 ** -11)
    assert np.array_equal(lv, -lv[::-1])
    assert np.array_equal(thr.astype(np.float64), 0.5 * (lv[:-1].astype(np.float64) + lv[1:].astype(np.float64)))


@pytest.mark.parametrize("bits", [2, 4])
def test_codes_are_nearest_level_of_the_rotated_coordinate(bits):
    """Brute force: every code is the nearest level of z = H(s x) / ||x|| (ties up)."""
    d = 64
    rng = np.random.default_rng(bits)
    x = rng.standard_normal((40, d)).astype(np.float16)
    words = np.array([0x9E3779B9, 0x7F4A7C15], dtype=np.int64)
    planes, n = tq.encode_tier(x, words, bits)
    k = tq.codes_from_tier_planes(planes, d, bits)
    lv, _ = tq.codebook(1 << bits)
    s = tq.signs_from_words(words, d)
    z = tq.fwht(x.astype(np.float64) * s) / np.linalg.norm(x.astype(np.float64), axis=1, keepdims=True)
    dist = np.abs(z[..., None] - lv.astype(np.float64)[None, None, :])
    best = dist.min(axis=-1)
    # the stored level is at the minimum distance (fp32 vs float64 rounding of z aside)
    assert np.all(dist[np.arange(40)[:, None], np.arange(d)[None, :], k] <= best + 1e-5)


def test_plane_layouts_bit_by_bit():
    """Hand-built level indices land at the documented bits of each tier's plane."""
    d = 32
    # TQ4: k -> sign = k >= 8, m = k - 8 or 7 - k; field (sign << 3) | m, element i at
    # bits 4 (i % 2) of byte i / 2
    k4 = np.array([[15, 0, 8, 7, 12, 3] + [7] * 26])
    sign = (k4 >= 8).astype(np.uint8)
    mag = np.where(k4 >= 8, k4 - 8, 7 - k4).astype(np.uint8)
    assert mag[0, :6].tolist() == [7, 7, 0, 0, 4, 4] and sign[0, :6].tolist() == [1, 0, 1, 0, 1, 0]
    p4 = tq.pack_bits((sign << 3) | mag, 4)
    assert p4.shape == (1, d // 2)
    assert p4[0, :3].tolist() == [0xF | 0x7 << 4, 0x8 | 0x0 << 4, 0xC | 0x4 << 4]
    assert np.array_equal(tq.codes_from_tier_planes((p4,), d, 4), k4)
    # TQ2: field (sign << 1) | m, element i at bits 2 (i % 4) of byte i / 4
    k2 = np.array([[3, 0, 2, 1, 1, 3, 0, 2] + [1] * 24])
    sign2 = (k2 >= 2).astype(np.uint8)
    mag2 = np.where(k2 >= 2, k2 - 2, 1 - k2).astype(np.uint8)
    p2 = tq.pack_bits((sign2 << 1) | mag2, 2)
    assert p2.shape == (1, d // 4)
    assert p2[0, 0] == (0b11 | 0b01 << 2 | 0b10 << 4 | 0b00 << 6)
    assert p2[0, 1] == (0b00 | 0b11 << 2 | 0b01 << 4 | 0b10 << 6)
    assert np.array_equal(tq.codes_from_tier_planes((p2,), d, 2), k2)
    # the encoder writes one such plane per tier, and reading it back gives the level
    # index it quantised to
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, d)).astype(np.float16)
    w = np.array([0x12345678], dtype=np.int64)
    for bits in (2, 4):
        planes, _ = tq.encode_tier(x, w, bits)
        assert len(planes) == 1 and planes[0].shape == (3, d * bits // 8)
        k, _ = tq.level_index(x, w, 1 << bits)
        assert np.array_equal(tq.codes_from_tier_planes(planes, d, bits), k)


def test_distortion_ladder_and_bytes_per_value():
    """More bits, less error (the tier ladder); storage as documented."""
    d = 128
    rng = np.random.default_rng(9)
    x = rng.standard_normal((256, d)).astype(np.float16)
    words = np.arange(d // 32, dtype=np.int64) * 0x2545F491 + 7
    err = {}
    for bits in (2, 3, 4):
        planes, n = tq.encode_tier(x, words, bits)
        xh = tq.decode_tier(planes, n, words, d, bits)
        err[bits] = float(np.mean((xh - x.astype(np.float64)) ** 2) / np.mean(x.astype(np.float64) ** 2))
    # relative MSE close to the Gaussian quantiser's (the rotated coordinates are ~N(0,1))
    assert abs(err[2] - 0.1175) < 0.02 and abs(err[3] - 0.03454) < 0.006 and abs(err[4] - 0.009497) < 0.002
    assert err[2] > err[3] > err[4]
    assert tq.bytes_per_value(d, 2) == (d // 4 + 2) / d
    assert tq.bytes_per_value(d, 4) == (d // 2 + 2) / d


def test_bytes_per_value_against_the_pages_table():
    """turbo2 matches the pages' bpv; turbo4 is exactly one fp16 per vector smaller."""
    rows = {r[1]: (float(r[2]), int(r[3])) for r in golden_rows("polykv_storage_and_roundtrip.txt")
            if r[0] == "bytes_per_value"}
    val, dec = rows["turbo2"]
    assert abs(tq.bytes_per_value(128, 2) - val) <= 0.5 * 10 ** -dec
    val, dec = rows["turbo4"]
    assert abs(tq.bytes_per_value(128, 4) + 2.0 / 128 - val) <= 0.5 * 10 ** -dec
