"""Pins of the block-diagonal, two-sign TurboQuant rotation (the form the PolyKV
page's fork runs: "S2 perf-path Level B" and its head_dim-512 note) against a dense
matrix built from scipy's Hadamard matrix, its orthogonality, nearest-level codes and
the first form it generalises."""

import numpy as np
import pytest
from scipy.linalg import block_diag, hadamard

from oracle import turboquant as tq

ROTS = [(256, 128), (512, 128), (128, 128), (512, 256), (64, 32)]


def _words(d, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << 32, size=d // 32, dtype=np.int64)


def _dense_r(d, g, w1, w2):
    """R = diag(s2) blockdiag(H_g) diag(s1) / sqrt(g) as a dense float64 matrix."""
    hb = block_diag(*([hadamard(g).astype(np.float64)] * (d // g)))
    s1 = tq.signs_from_words(w1, d)
    s2 = np.ones(d) if w2 is None else tq.signs_from_words(w2, d)
    return (s2[:, None] * hb * s1[None, :]) / np.sqrt(g)


@pytest.mark.parametrize("d,g", ROTS)
def test_dense_rotation_is_orthogonal(d, g):
    r = _dense_r(d, g, _words(d, 1), _words(d, 2))
    assert np.allclose(r @ r.T, np.eye(d), atol=1e-12)


@pytest.mark.parametrize("d,g", ROTS)
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codes_are_nearest_level_of_dense_rotation(d, g, bits):
    """Every code is the nearest level of z = sqrt(D) R x / ||x|| (fp32 rounding aside)."""
    rng = np.random.default_rng(d + g + bits)
    x = rng.standard_normal((30, d)).astype(np.float16)
    w1, w2 = _words(d, 3), _words(d, 4)
    rot = tq.Rotation(w1, w2, g)
    planes, _ = tq.encode_tier(x, rot, bits)
    k = tq.codes_from_tier_planes(planes, d, bits)
    lv, _ = tq.codebook(1 << bits)
    xd = x.astype(np.float64)
    z = np.sqrt(d) * (xd @ _dense_r(d, g, w1, w2).T) / np.linalg.norm(xd, axis=1, keepdims=True)
    dist = np.abs(z[..., None] - lv.astype(np.float64)[None, None, :])
    got = np.take_along_axis(dist, k[..., None], axis=-1)[..., 0]
    assert np.all(got <= dist.min(axis=-1) + 1e-5)


@pytest.mark.parametrize("d,g", ROTS)
def test_decode_equals_dense_inverse(d, g):
    """x_hat = n R^T c[k] / sqrt(D), computed with the dense matrix."""
    rng = np.random.default_rng(7 * d + g)
    x = rng.standard_normal((20, d)).astype(np.float16)
    w1, w2 = _words(d, 5), _words(d, 6)
    rot = tq.Rotation(w1, w2, g)
    for bits in (2, 3, 4):
        planes, n = tq.encode_tier(x, rot, bits)
        lv, _ = tq.codebook(1 << bits)
        c = lv.astype(np.float64)[tq.codes_from_tier_planes(planes, d, bits)]
        want = n.astype(np.float64)[:, None] * (c @ _dense_r(d, g, w1, w2)) / np.sqrt(d)
        assert np.allclose(tq.decode_tier(planes, n, rot, d, bits), want, rtol=0, atol=1e-12)


def test_first_form_is_the_default_rotation():
    d = 256
    x = np.random.default_rng(8).standard_normal((50, d)).astype(np.float16)
    w = _words(d, 9)
    for bits in (2, 3, 4):
        a, na = tq.encode_tier(x, w, bits)
        b, nb = tq.encode_tier(x, tq.Rotation(w, None, None), bits)
        c, nc = tq.encode_tier(x, tq.Rotation(w, None, d), bits)
        for pa, pb, pc in zip(a, b, c):
            assert np.array_equal(pa, pb) and np.array_equal(pa, pc)
        assert np.array_equal(na, nb) and np.array_equal(na, nc)


@pytest.mark.parametrize("d,g", [(512, 128), (256, 128)])
def test_block_rotation_distortion_matches_gaussian_quantiser(d, g):
    """Decoded rows keep the Gaussian quantiser's relative MSE (the block transform
    still spreads each row's energy evenly)."""
    rng = np.random.default_rng(d)
    x = rng.standard_normal((200, d)).astype(np.float16)
    rot = tq.Rotation(_words(d, 10), _words(d, 11), g)
    planes, n = tq.encode_tier(x, rot, 3)
    xh = tq.decode_tier(planes, n, rot, d, 3)
    xd = x.astype(np.float64)
    err = float(np.mean((xh - xd) ** 2) / np.mean(xd ** 2))
    assert abs(err - 0.03454) < 0.006


def test_block_width_must_divide_head_dim():
    x = np.zeros((1, 128), dtype=np.float16)
    with pytest.raises(ValueError):
        tq.encode_tier(x, tq.Rotation(_words(128, 1), None, 96), 3)
    with pytest.raises(ValueError):
        tq.encode_tier(x, tq.Rotation(_words(128, 1), None, 256), 3)


@pytest.mark.parametrize("d,g", ROTS)
def test_rotated_query_identity(d, g):
    """q . x_hat = (n / sqrt(D)) (R q) . c[k]: a TurboQuant K can be read in the rotated
    domain against the rotated query (PolyKV page, "S2 perf-path Level B")."""
    rng = np.random.default_rng(d * 3 + g)
    k = rng.standard_normal((25, d)).astype(np.float16)
    q = rng.standard_normal((4, d))
    w1, w2 = _words(d, 12), _words(d, 13)
    rot = tq.Rotation(w1, w2, g)
    r = _dense_r(d, g, w1, w2)
    for bits in (2, 3, 4):
        planes, n = tq.encode_tier(k, rot, bits)
        lv, _ = tq.codebook(1 << bits)
        c = lv.astype(np.float64)[tq.codes_from_tier_planes(planes, d, bits)]
        direct = q @ tq.decode_tier(planes, n, rot, d, bits).T
        rotated = ((q @ r.T) @ c.T) * n.astype(np.float64)[None, :] / np.sqrt(d)
        assert np.allclose(direct, rotated, rtol=0, atol=1e-11)
