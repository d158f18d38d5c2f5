"""Pins of the q8_0 oracle against definitions it does not share code with."""

import numpy as np
import pytest

from oracle import q8_0
from tests.conftest import golden_rows


def _rand_rows(rng, rows, d, outliers=True):
    x = rng.standard_normal((rows, d)).astype(np.float32)
    if outliers:
        ch = rng.choice(d, size=4, replace=False)
        x[:, ch] *= 20.0
    return x.astype(np.float16)


@pytest.mark.parametrize("d", [32, 64, 128, 512])
def test_roundtrip_error_bound(d):
    rng = np.random.default_rng(1)
    x = _rand_rows(rng, 300, d)
    codes, scales = q8_0.encode(x)
    xh = q8_0.decode(codes, scales)
    d16 = np.repeat(scales.astype(np.float64), 32, axis=-1)
    err = np.abs(x.astype(np.float64) - xh)
    # |x - q d16| <= d16 / 2, plus the f32 division's rounding (|x/d16| <= 127.1)
    assert np.all(err <= d16 * (0.5 + 2.0 ** -17))


def test_codes_are_nearest_integer_multiple_of_stored_scale():
    """Brute force: the code is the integer q in [-127, 127] nearest to x / d16."""
    rng = np.random.default_rng(2)
    x = _rand_rows(rng, 64, 128)
    codes, scales = q8_0.encode(x)
    xb = x.astype(np.float64).reshape(64, 4, 32)
    d16 = scales.astype(np.float64)
    cand = np.arange(-127, 128, dtype=np.float64)
    checked = 0
    for r in range(64):
        for b in range(4):
            for j in range(32):
                t = xb[r, b, j] / d16[r, b]
                frac = abs(t) - np.floor(abs(t))
                if abs(frac - 0.5) < 1e-5:  # near a tie: the f32 rounding decides
                    continue
                best = cand[np.argmin(np.abs(cand - t))]
                assert codes[r, b * 32 + j] == best
                checked += 1
    assert checked > 8000


def test_ties_round_half_away_from_zero():
    # amax = 127 gives d32 = 1 exactly, so x / d16 = x and halves are exact ties.
    blk = np.zeros(32, dtype=np.float16)
    blk[0] = 127.0
    blk[1] = 2.5
    blk[2] = -2.5
    blk[3] = 0.5
    blk[4] = -0.5
    blk[5] = 3.5
    blk[6] = -126.5
    codes, scales = q8_0.encode(blk[None])
    assert float(scales[0, 0]) == 1.0
    assert list(codes[0, :7]) == [127, 3, -3, 1, -1, 4, -127]


def test_extremes_and_zero_block():
    x = np.zeros((2, 64), dtype=np.float16)
    x[1, 32] = -7.0  # block 1 of row 1: amax 7, the element itself maps to -127
    codes, scales = q8_0.encode(x)
    assert np.all(codes[0] == 0) and np.all(scales[0] == 0)
    assert codes[1, 32] == -127
    assert float(scales[1, 1]) == float(np.float16(np.float32(7.0) / np.float32(127.0)))
    assert np.all(codes[1, :32] == 0) and float(scales[1, 0]) == 0.0


def test_hand_block():
    # amax 63.5 -> d32 = 0.5 exactly; codes are x / 0.5 rounded.
    vals = [63.5, -1.25, 0.75, 0.2, -0.3, 10.0]
    blk = np.zeros(32, dtype=np.float16)
    blk[: len(vals)] = vals
    codes, scales = q8_0.encode(blk[None])
    assert float(scales[0, 0]) == 0.5
    assert list(codes[0, :6]) == [127, -3, 2, 0, -1, 20]


def test_bytes_per_value_matches_pages():
    rows = {r[1]: (float(r[2]), int(r[3])) for r in golden_rows("polykv_storage_and_roundtrip.txt")
            if r[0] == "bytes_per_value"}
    val, dec = rows["q8_0"]
    assert abs(q8_0.bytes_per_value(128) - val) <= 0.5 * 10 ** -dec + 1e-12


def test_scales_at_the_bottom_of_the_fp16_range():
    """absmax / 127 below half the smallest fp16 subnormal (2^-25) rounds to a zero
    scale: the block stores zero codes and decodes to zeros, so its error is |x| itself
    (< 127 * 2^-25), not d16 / 2.  With absmax = 2^-17 the scale rounds up to the
    smallest subnormal, 2^-24, so x / d16 = +-128: the codes clamp to +-127 (never
    -128), and the error, one d16, exceeds d16 / 2.  The d16 / 2 bound needs a normal
    d16, whose rounding moves it by at most 2^-11 relative."""
    tiny = np.float16(2.0 ** -20)  # absmax / 127 ~ 7.5e-9 < 2^-25 ~ 3.0e-8
    blk = np.zeros((2, 32), dtype=np.float16)
    blk[0, 0], blk[0, 7] = tiny, -tiny / np.float16(2)
    blk[1, 0], blk[1, 1] = np.float16(2.0 ** -17), np.float16(-(2.0 ** -17))
    codes, scales = q8_0.encode(blk)
    assert float(scales[0, 0]) == 0.0 and not codes[0].any()
    assert np.all(q8_0.decode(codes, scales)[0] == 0.0)
    assert float(scales[1, 0]) == 2.0 ** -24
    assert codes[1, 0] == 127 and codes[1, 1] == -127
    err = np.abs(q8_0.decode(codes, scales)[1, :2] - blk[1, :2].astype(np.float64))
    assert np.all(err == 2.0 ** -24)
