"""GPU encoders vs the oracle: codes, scales, planes and norms must be bit-exact."""

import numpy as np
import pytest
import torch

import synth
from oracle import q8_0 as oq8
from oracle import turboquant as otq

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qps():
    import quantized_position_split_gb300 as q
    from quantized_position_split_gb300 import build
    build.build()
    return q


def _rows(n, d, seed, outliers=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, d), generator=g)
    if outliers:
        ch = torch.randperm(d, generator=g)[:4]
        x[:, ch] *= 20
    x[3] = 0  # a zero row
    x[5, :32] = 0  # a zero block
    return x.half()


@pytest.mark.parametrize("d", [32, 64, 128, 256, 512])
def test_q8_0_bit_exact(qps, d):
    x = _rows(1000 + 3, d, d)
    codes, scales = qps.kv_quant_q8_0(x.cuda())
    rc, rs = oq8.encode(x.numpy())
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), rs.view(np.uint16))


def test_q8_0_every_fp16_value_for_fixed_amax(qps):
    """For amax in a few values, every finite fp16 x with |x| <= amax, one block each
    31 values plus the amax element."""
    allv = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    allv = allv[np.isfinite(allv)]
    # 2^-17: the scale rounds to the smallest subnormal and the codes clamp at +-127;
    # 2^-20: the scale rounds to zero and the block stores zeros
    for amax in [1.0, 3.140625, 0.0009765625, 65504.0, 2.0 ** -17, 2.0 ** -20]:
        vals = allv[np.abs(allv.astype(np.float64)) <= amax]
        pad = (-len(vals)) % 31
        vals = np.concatenate([vals, np.zeros(pad, dtype=np.float16)]).reshape(-1, 31)
        blocks = np.concatenate([np.full((vals.shape[0], 1), amax, dtype=np.float16), vals], axis=1)
        x = torch.from_numpy(blocks.copy())
        codes, scales = qps.kv_quant_q8_0(x.cuda())
        rc, rs = oq8.encode(blocks)
        assert np.array_equal(codes.cpu().numpy(), rc), amax
        assert np.array_equal(scales.cpu().numpy().view(np.uint16), rs.view(np.uint16)), amax


@pytest.mark.parametrize("d", [32, 64, 128, 256, 512])
def test_tq3_bit_exact(qps, d):
    x = _rows(2000 + 5, d, 100 + d, outliers=(d != 64))
    words = synth.sign_bits(d, 42)
    lo2, hi1, n = qps.kv_quant_tq3(x.cuda(), words)
    rlo, rhi, rn = otq.encode(x.numpy(), words.numpy())
    glo, ghi, gn = lo2.cpu().numpy(), hi1.cpu().numpy(), n.cpu().numpy()
    assert np.array_equal(gn.view(np.uint16), rn.view(np.uint16))
    bad = np.nonzero((glo != rlo).any(-1) | (ghi != rhi).any(-1))[0]
    if bad.size:
        # report how close the disagreeing coordinates were to a threshold
        _, thr = otq.codebook()
        xr = x.numpy()[bad[:4]].astype(np.float64)
        s = otq.signs_from_words(words.numpy(), d)
        z = otq.fwht(xr * s) / np.linalg.norm(xr, axis=1, keepdims=True)
        dist = np.min(np.abs(z[..., None] - thr.astype(np.float64)), axis=-1).min()
        pytest.fail(f"{bad.size} rows differ; nearest threshold distance {dist:.3e}")


@pytest.mark.parametrize("d", [32, 64, 128, 256, 512])
@pytest.mark.parametrize("bits", [2, 4])
def test_tq_tier_bit_exact(qps, d, bits):
    """TQ2 / TQ4 fields and norms equal the oracle's, zero row and zero block included."""
    x = _rows(2000 + 5, d, 200 + d + bits, outliers=(d != 64))
    words = synth.sign_bits(d, 42)
    enc = qps.kv_quant_tq2 if bits == 2 else qps.kv_quant_tq4
    codes, n = enc(x.cuda(), words)
    (rc,), rn = otq.encode_tier(x.numpy(), words.numpy(), bits)
    assert codes.shape == (x.shape[0], d * bits // 8)
    assert np.array_equal(n.cpu().numpy().view(np.uint16), rn.view(np.uint16))
    bad = np.nonzero((codes.cpu().numpy() != rc).any(-1))[0]
    if bad.size:
        _, thr = otq.codebook(1 << bits)
        xr = x.numpy()[bad[:4]].astype(np.float64)
        s = otq.signs_from_words(words.numpy(), d)
        z = otq.fwht(xr * s) / np.linalg.norm(xr, axis=1, keepdims=True)
        dist = np.min(np.abs(z[..., None] - thr.astype(np.float64)), axis=-1).min()
        pytest.fail(f"{bad.size} rows differ; nearest threshold distance {dist:.3e}")
    assert not codes[3].any() and float(n[3]) == 0.0  # the zero row


@pytest.mark.parametrize("d,g", [(512, 128), (256, 128), (128, 32), (64, 64)])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_tq_rotation_bit_exact(qps, d, g, bits):
    """The block-diagonal two-sign rotation: planes and norms equal the oracle's."""
    x = _rows(1500 + 3, d, 300 + d + g + bits, outliers=(d != 64))
    w1, w2 = synth.sign_bits(d, 42), synth.sign_bits(d, 43)
    planes = qps.encode_kv(f"tq{bits}", x.cuda().reshape(-1, 1, d), qps.Rotation(w1, w2, g)).planes
    rp, rn = otq.encode_tier(x.numpy(), otq.Rotation(w1.numpy(), w2.numpy(), g), bits)
    assert np.array_equal(planes[-1].cpu().numpy().reshape(-1).view(np.uint16), rn.view(np.uint16))
    for got, want in zip(planes[:-1], rp):
        assert np.array_equal(got.cpu().numpy().reshape(want.shape), want)


def test_tq3_sign_vector_changes_codes(qps):
    x = _rows(64, 128, 7, outliers=False).cuda()
    a = qps.kv_quant_tq3(x, synth.sign_bits(128, 42))[0]
    b = qps.kv_quant_tq3(x, synth.sign_bits(128, 43))[0]
    assert not torch.equal(a, b)


def test_encoders_row_stride(qps):
    x = _rows(300, 256, 9)
    xs = x[:, :128]  # a strided view: row stride 256, head_dim 128
    c1, s1 = qps.kv_quant_q8_0(x.cuda()[:, :128])
    rc, rs = oq8.encode(xs.contiguous().numpy())
    assert np.array_equal(c1.cpu().numpy(), rc)
    words = synth.sign_bits(128, 42)
    lo2, hi1, n = qps.kv_quant_tq3(x.cuda()[:, :128], words)
    rlo, rhi, rn = otq.encode(xs.contiguous().numpy(), words.numpy())
    assert np.array_equal(lo2.cpu().numpy(), rlo) and np.array_equal(hi1.cpu().numpy(), rhi)


@pytest.mark.parametrize("d", [32, 128, 512])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_tq_exact_ties_bit_exact(qps, d, bits):
    """Rows whose rotated coordinates sit exactly on the middle threshold, 0: with
    x = c s_i e_i + c s_j e_j the sign diagonal is undone, H (s * x) is +-2c at half the
    coordinates and exactly 0 at the other half.  The oracle puts a coordinate on a
    threshold in the upper cell; the GPU encoders must agree bit for bit."""
    words = synth.sign_bits(d, 42)
    s = otq.signs_from_words(words.numpy(), d)
    rng = np.random.default_rng(1000 + d + bits)
    x = np.zeros((64, d))
    for r in range(64):
        i, j = rng.choice(d, 2, replace=False)
        c = 2.0 ** int(rng.integers(-6, 7))
        x[r, i], x[r, j] = s[i] * c, s[j] * c
    x16 = x.astype(np.float16)
    planes, rn = otq.encode_tier(x16, words.numpy(), bits)
    k = otq.codes_from_tier_planes(planes, d, bits)
    assert (k == (1 << bits) // 2).sum() >= 64 * d // 2  # the ties took the upper cell
    xt = torch.from_numpy(x16).cuda()
    if bits == 3:
        lo2, hi1, n = qps.kv_quant_tq3(xt, words)
        got = (lo2.cpu().numpy(), hi1.cpu().numpy())
    else:
        codes, n = (qps.kv_quant_tq2 if bits == 2 else qps.kv_quant_tq4)(xt, words)
        got = (codes.cpu().numpy(),)
    assert np.array_equal(n.cpu().numpy().view(np.uint16), rn.view(np.uint16))
    for g, want in zip(got, planes):
        assert np.array_equal(g, want)
