"""Pins of the whole-layer references (oracle.pipeline): K and V are read through their
stored formats, and a layer reference is plain attention over those rows.

The dequantised rows are characterised without the oracle's own decoders: a q8_0 row
lies on its blocks' grids (the stored fp16 scale times the nearest integer in
[-127, 127]); a TurboQuant row, rotated by a dense matrix built from scipy's Hadamard
matrix, sits exactly on the codebook levels times norm / sqrt(D), at the level nearest
to the input's own rotated coordinate.
"""

import numpy as np
import pytest
import scipy.linalg
import torch

import synth
from oracle import pipeline
from oracle import turboquant as tq


def _rows(seed, n, d, outliers=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, d))
    if outliers:
        x[:, rng.choice(d, size=4, replace=False)] *= 20.0
    return x.astype(np.float16)


def test_f16_is_read_as_stored():
    x = _rows(1, 33, 64)
    assert np.array_equal(pipeline.dequant("f16", x), x.astype(np.float64))


@pytest.mark.parametrize("d", [32, 128, 512])
def test_q8_0_rows_lie_on_their_block_grids(d):
    x = _rows(2, 50, d, outliers=True)
    got = pipeline.dequant("q8_0", x)
    xb = x.astype(np.float64).reshape(50, d // 32, 32)
    amax = np.max(np.abs(x.astype(np.float32).reshape(50, d // 32, 32)), axis=-1)
    d16 = (amax / np.float32(127.0)).astype(np.float16).astype(np.float64)[..., None]
    q = got.reshape(50, d // 32, 32) / d16
    assert np.array_equal(q, np.round(q)) and np.max(np.abs(q)) <= 127
    err = np.abs(xb - got.reshape(xb.shape))
    # nearest grid point: only a neighbour at least as close is tolerated (ties)
    assert np.all(err <= d16 * (0.5 + 2.0 ** -17))
    assert np.max(err) > 0  # it was quantised


@pytest.mark.parametrize("fmt", ["tq2", "tq3", "tq4"])
@pytest.mark.parametrize("d", [64, 128])
def test_turboquant_rows_rotate_onto_the_nearest_levels(fmt, d):
    bits = int(fmt[2])
    words = synth.sign_bits(d, 42).numpy()
    x16 = _rows(3 + d + bits, 40, d)
    got = pipeline.dequant(fmt, x16, words)
    s = tq.signs_from_words(words, d)
    rot = scipy.linalg.hadamard(d).astype(np.float64) * s[None, :] / np.sqrt(d)  # R = H diag(s) / sqrt(D)
    x = x16.astype(np.float64)
    nrm = np.linalg.norm(x, axis=1, keepdims=True)
    n16 = pipeline.encode(fmt, x16, words)[-1].astype(np.float64)[:, None]  # the stored norm plane
    assert np.allclose(n16, nrm, rtol=2.0 ** -10, atol=0)
    w = np.sqrt(d) * (got @ rot.T) / n16  # must be codebook levels
    levels, thr = tq.codebook(1 << bits)
    lv = levels.astype(np.float64)
    idx = np.argmin(np.abs(w[..., None] - lv), axis=-1)
    assert np.allclose(w, lv[idx], atol=1e-9)
    z = np.sqrt(d) * (x @ rot.T) / nrm
    near_tie = np.min(np.abs(z[..., None] - thr.astype(np.float64)), axis=-1) < 1e-5
    nearest = np.argmin(np.abs(z[..., None] - lv), axis=-1)
    assert np.array_equal(idx[~near_tie], nearest[~near_tie])


@pytest.mark.parametrize("k_fmt,v_fmt", [("f16", "f16"), ("q8_0", "q8_0"), ("q8_0", "tq3"), ("tq4", "tq4")])
def test_layer_reference_is_sdpa_over_the_stored_rows(k_fmt, v_fmt):
    """Against torch's float64 SDPA (GQA by repeating KV heads) over the rows the
    formats store, characterised by the pins above."""
    n, hq, hkv, d = 57, 6, 2, 64
    words = synth.sign_bits(d, 42).numpy()
    q = _rows(10, hq, d).reshape(1, hq, d)
    k = _rows(11, n * hkv, d, outliers=True).reshape(n, hkv, d)
    v = _rows(12, n * hkv, d).reshape(n, hkv, d)
    o, lse = pipeline.layer_reference(q, k, v, k_fmt, v_fmt, 0.125, 0.0, words)
    kh = pipeline.dequant(k_fmt, k, words)
    vh = pipeline.dequant(v_fmt, v, words)
    if k_fmt != "f16":
        assert not np.array_equal(kh, k.astype(np.float64))
    if v_fmt != "f16":
        assert not np.array_equal(vh, v.astype(np.float64))
    g = hq // hkv
    kt = torch.from_numpy(np.repeat(kh.transpose(1, 0, 2), g, axis=0))
    vt = torch.from_numpy(np.repeat(vh.transpose(1, 0, 2), g, axis=0))
    qt = torch.from_numpy(q.astype(np.float64).transpose(1, 0, 2))
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.125)
    assert np.allclose(o[0], ref[:, 0, :].numpy(), rtol=0, atol=1e-12)
    s = np.einsum("hd,hnd->hn", qt[:, 0].numpy(), kt.numpy()) * 0.125
    m = s.max(axis=1)
    assert np.allclose(lse[0], m + np.log(np.exp(s - m[:, None]).sum(axis=1)), atol=1e-12)
