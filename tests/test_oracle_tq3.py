"""Pins of the FWHT and the TQ3 encoder / decoder."""

import numpy as np
import pytest
import scipy.linalg

import synth
from oracle import turboquant as tq
from tests.conftest import golden_rows


def _signs(d):
    return synth.sign_bits(d, 42).numpy()


@pytest.mark.parametrize("d", [2, 4, 8, 32, 64, 128, 256, 512])
def test_fwht_equals_scipy_hadamard(d):
    eye = np.eye(d)
    h = tq.fwht(eye)  # row i = H e_i (H symmetric)
    assert np.array_equal(h, scipy.linalg.hadamard(d).astype(np.float64))
    assert np.array_equal(h @ h.T, d * np.eye(d))


def test_fwht_equals_sylvester_recursion():
    h = np.array([[1.0]])
    while h.shape[0] < 256:
        h = np.block([[h, h], [h, -h]])
    x = np.random.default_rng(0).standard_normal((5, 256))
    assert np.allclose(tq.fwht(x), x @ h.T, atol=1e-10)


def test_fwht_float32_exact_on_small_integers():
    x = np.random.default_rng(1).integers(-8, 8, size=(7, 128)).astype(np.float32)
    assert np.array_equal(tq.fwht(x, np.float32).astype(np.float64), tq.fwht(x.astype(np.float64)))


@pytest.mark.parametrize("d", [64, 128, 512])
def test_rotation_is_orthonormal_and_parseval(d):
    s = tq.signs_from_words(_signs(d), d)
    r = scipy.linalg.hadamard(d) @ np.diag(s) / np.sqrt(d)
    assert np.allclose(r @ r.T, np.eye(d), atol=1e-12)
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal((2, d))
    rq = tq.fwht(s * q) / np.sqrt(d)
    rk = tq.fwht(s * k) / np.sqrt(d)
    assert np.isclose(np.linalg.norm(rq), np.linalg.norm(q), rtol=1e-13)
    assert np.isclose(rq @ rk, q @ k, rtol=1e-12, atol=1e-12)
    # inverse is the transpose
    assert np.allclose(s * tq.fwht(rq) / np.sqrt(d), q, atol=1e-12)


def test_sign_word_bit_order():
    words = np.array([0b101, 1 << 31], dtype=np.int64)
    s = tq.signs_from_words(words, 64)
    neg = set(np.nonzero(s < 0)[0].tolist())
    assert neg == {0, 2, 63}


def test_pack_bit_positions():
    vals = np.zeros(32, dtype=np.uint8)
    vals[5] = 2  # byte 1, bits 2..3
    vals[31] = 3  # byte 7, bits 6..7
    p = tq.pack_bits(vals[None], 2)[0]
    assert p[1] == 2 << 2 and p[7] == 3 << 6 and p.sum() == (2 << 2) + (3 << 6)
    bits = np.zeros(32, dtype=np.uint8)
    bits[9] = 1
    p1 = tq.pack_bits(bits[None], 1)[0]
    assert p1[1] == 2 and p1.sum() == 2
    rng = np.random.default_rng(5)
    v = rng.integers(0, 4, size=(3, 128)).astype(np.uint8)
    assert np.array_equal(tq.unpack_bits(tq.pack_bits(v, 2), 2, 128), v)


@pytest.mark.parametrize("d", [64, 128, 512])
def test_codes_are_nearest_level_of_rotated_coordinate(d):
    """Independent float64 recomputation with scipy's Hadamard matrix."""
    rng = np.random.default_rng(6)
    x16 = rng.standard_normal((40, d)).astype(np.float16)
    words = _signs(d)
    lo2, hi1, n16 = tq.encode(x16, words)
    k = tq.codes_from_planes(lo2, hi1, d)
    s = tq.signs_from_words(words, d)
    x = x16.astype(np.float64)
    z = (x * s) @ scipy.linalg.hadamard(d).T / np.linalg.norm(x, axis=1, keepdims=True)
    levels, thr = tq.codebook()
    nearest = np.argmin(np.abs(z[..., None] - levels.astype(np.float64)), axis=-1)
    near_tie = np.min(np.abs(z[..., None] - thr.astype(np.float64)), axis=-1) < 1e-5
    assert np.array_equal(k[~near_tie], nearest[~near_tie])
    assert np.allclose(n16.astype(np.float64), np.linalg.norm(x, axis=1), rtol=2 ** -10)


@pytest.mark.parametrize("d", [128, 512])
def test_roundtrip_distortion_and_pages_cosine(d):
    rng = np.random.default_rng(7)
    x16 = rng.standard_normal((2000, d)).astype(np.float16)
    words = _signs(d)
    xh = tq.decode(*tq.encode(x16, words), words, d)
    x = x16.astype(np.float64)
    rel = np.sum((x - xh) ** 2) / np.sum(x ** 2)
    assert abs(rel - 0.03455) < 2.5e-3
    cos = np.mean(np.sum(x * xh, 1) / np.linalg.norm(x, axis=1) / np.linalg.norm(xh, axis=1))
    row = [r for r in golden_rows("polykv_storage_and_roundtrip.txt") if r[0] == "roundtrip_cosine"][0]
    assert abs(cos - float(row[2])) <= 0.5 * 10 ** -int(row[3]) + 1e-3


def test_decode_matches_explicit_matrix():
    d = 128
    rng = np.random.default_rng(8)
    x16 = rng.standard_normal((9, d)).astype(np.float16)
    words = _signs(d)
    lo2, hi1, n16 = tq.encode(x16, words)
    levels, _ = tq.codebook()
    ck = levels.astype(np.float64)[tq.codes_from_planes(lo2, hi1, d)]
    s = tq.signs_from_words(words, d)
    want = (n16.astype(np.float64)[:, None] / d) * (ck @ scipy.linalg.hadamard(d).T) * s
    assert np.allclose(tq.decode(lo2, hi1, n16, words, d), want, atol=1e-12)


def test_power_of_two_scale_invariance_and_zero_row():
    d = 128
    rng = np.random.default_rng(9)
    x16 = rng.standard_normal((16, d)).astype(np.float16)
    words = _signs(d)
    a = tq.encode(x16, words)
    b = tq.encode((x16.astype(np.float32) * 4).astype(np.float16), words)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.array_equal(a[2].astype(np.float32) * 4, b[2].astype(np.float32))
    z = tq.encode(np.zeros((1, d), dtype=np.float16), words)
    assert not z[0].any() and not z[1].any() and float(z[2][0]) == 0.0


def test_bytes_per_value_matches_pages():
    row = [r for r in golden_rows("polykv_storage_and_roundtrip.txt")
           if r[0] == "bytes_per_value" and r[1] == "turbo3"][0]
    assert abs(tq.bytes_per_value(128) - float(row[2])) <= 0.5 * 10 ** -int(row[3])


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("d", [32, 128, 512])
def test_exact_tie_takes_the_upper_cell(d, bits):
    """With every sign +1, x = e_0 + e_1 gives H x = 2 at the even and exactly 0 at the
    odd coordinates (column 0 of H is all ones, column 1 alternates in sign).  0 is the
    threshold between the two middle levels of every symmetric codebook, so the odd
    coordinates sit exactly on a threshold and must take the upper cell, index L / 2;
    the even ones (z = sqrt 2, away from every threshold) take the nearest level."""
    n_levels = 1 << bits
    x16 = np.zeros((1, d), dtype=np.float16)
    x16[0, :2] = 1.0
    words = np.zeros(d // 32, dtype=np.uint32)  # s = +1 everywhere
    levels, thr = tq.codebook(n_levels)
    assert thr[n_levels // 2 - 1] == 0.0
    planes, n16 = tq.encode_tier(x16, words, bits)
    k = tq.codes_from_tier_planes(planes, d, bits)[0]
    assert np.all(k[1::2] == n_levels // 2)
    assert np.min(np.abs(thr.astype(np.float64) - np.sqrt(2.0))) > 1e-2
    assert np.all(k[0::2] == np.argmin(np.abs(levels.astype(np.float64) - np.sqrt(2.0))))
