"""Pins of the attention / split / combine oracle: closed forms, library routines,
brute force and the split identity."""

import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

from oracle import attention as att
from oracle import pipeline


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_single_key_closed_form():
    rng = np.random.default_rng(0)
    q, k, v = _rand(rng, 3, 16), _rand(rng, 1, 16), _rand(rng, 1, 16)
    o, lse = att.attend(q, k, v, 0.25)
    assert np.allclose(o, np.repeat(v, 3, 0), atol=0)
    assert np.allclose(lse, 0.25 * (q @ k[0]), atol=1e-15)


def test_identical_keys_give_mean_and_log_n():
    rng = np.random.default_rng(1)
    n = 37
    q = _rand(rng, 2, 8)
    k = np.repeat(_rand(rng, 1, 8), n, 0)
    v = _rand(rng, n, 8)
    o, lse = att.attend(q, k, v, 0.5)
    assert np.allclose(o, np.repeat(v.mean(0, keepdims=True), 2, 0), atol=1e-14)
    assert np.allclose(lse, 0.5 * (q @ k[0]) + math.log(n), atol=1e-13)


def test_zero_query_is_uniform():
    rng = np.random.default_rng(2)
    k, v = _rand(rng, 50, 8), _rand(rng, 50, 8)
    o, lse = att.attend(np.zeros((1, 8)), k, v, 1.0)
    assert np.allclose(o[0], v.mean(0), atol=1e-14) and np.isclose(lse[0], math.log(50))


def test_empty_part():
    o, lse = att.attend(np.ones((2, 4)), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_gqa_decode_matches_torch_sdpa_and_scipy_logsumexp():
    rng = np.random.default_rng(3)
    hq, hkv, n, d = 8, 2, 70, 32
    q = _rand(rng, 1, hq, d)
    k = _rand(rng, n, hkv, d)
    v = _rand(rng, n, hkv, d)
    scale = 1 / math.sqrt(d)
    o, lse = att.gqa_decode(q, k, v, scale)
    tq = torch.tensor(q).unsqueeze(2)  # [1, hq, 1, d]
    tk = torch.tensor(k).permute(1, 0, 2).unsqueeze(0)  # [1, hkv, n, d]
    tv = torch.tensor(v).permute(1, 0, 2).unsqueeze(0)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale, enable_gqa=True)
    assert np.allclose(o, ref[:, :, 0, :].numpy(), atol=1e-13)
    g = hq // hkv
    for h in range(hq):
        logit = np.einsum("d,nd->n", q[0, h], k[:, h // g]) * scale
        assert np.isclose(lse[0, h], logsumexp(logit), atol=1e-13)


def test_gqa_group_mapping():
    hq, hkv, n, d = 8, 4, 5, 4
    q = np.ones((1, hq, d))
    k = np.zeros((n, hkv, d))
    v = np.zeros((n, hkv, d))
    for h in range(hkv):
        v[:, h, :] = h
    o, _ = att.gqa_decode(q, k, v, 1.0)
    assert np.array_equal(o[0, :, 0], np.array([h // 2 for h in range(hq)], dtype=float))


@pytest.mark.parametrize("softcap", [0.0, 2.0])
def test_split_equals_unsplit_for_every_window(softcap):
    rng = np.random.default_rng(4)
    n, d = 48, 16
    q = _rand(rng, 1, 4, d) * 2
    k = _rand(rng, n, 2, d)
    v = _rand(rng, n, 2, d)
    ref_o, ref_l = att.gqa_decode(q, k, v, 0.3, softcap)
    for wc in range(0, n + 1):
        tiles = [(a, min(a + 7, n)) for a in range(wc, n, 7)] or [(n, n)]
        o, l = att.split_decode(q, k, v, wc, 0.3, softcap, tail_tiles=tiles)
        assert np.allclose(o, ref_o, atol=1e-13) and np.allclose(l, ref_l, atol=1e-13), wc


@pytest.mark.parametrize("softcap", [0.0, 1.5])
def test_brute_force_loops(softcap):
    rng = np.random.default_rng(5)
    for n in range(1, 17):
        q, k, v = _rand(rng, 3, 6) * 3, _rand(rng, n, 6), _rand(rng, n, 5)
        o1, l1 = att.attend(q, k, v, 0.7, softcap)
        o2, l2 = att.attend_loops(q, k, v, 0.7, softcap)
        assert np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)


def test_softcap_bounds_limit_and_order():
    rng = np.random.default_rng(6)
    q, k, v = _rand(rng, 2, 8) * 10, _rand(rng, 30, 8) * 10, _rand(rng, 30, 8)
    s = att.logits(q, k, 1.0, 5.0)
    assert np.all(np.abs(s) <= 5.0) and np.max(np.abs(q @ k.T)) > 50.0
    o_inf, l_inf = att.attend(q, k, v, 1.0, 1e9)
    o_raw, l_raw = att.attend(q, k, v, 1.0, 0.0)
    assert np.allclose(o_inf, o_raw, atol=1e-9) and np.allclose(l_inf, l_raw, atol=1e-6)
    # capping the logits before the softmax is not the same as not capping them
    o_cap, l_cap = att.attend(q, k, v, 1.0, 5.0)
    assert np.max(np.abs(o_cap - o_raw)) > 1e-2
    # the capped result equals a softmax over explicitly capped logits
    capped = 5.0 * np.tanh((q @ k.T) / 5.0)
    w = np.exp(capped - capped.max(1, keepdims=True))
    assert np.allclose(o_cap, (w @ v) / w.sum(1, keepdims=True), atol=1e-13)
    assert np.allclose(l_cap, logsumexp(capped, axis=1), atol=1e-13)


def test_combine_identities():
    rng = np.random.default_rng(7)
    o = _rand(rng, 5, 3, 4)
    l = _rand(rng, 5, 3)
    l[2, 1] = -np.inf
    o_all, l_all = att.lse_combine(o, l)
    # nested combination equals one combination
    a = att.lse_combine(o[:2], l[:2])
    b = att.lse_combine(o[2:], l[2:])
    o_n, l_n = att.lse_combine(np.stack([a[0], b[0]]), np.stack([a[1], b[1]]))
    assert np.allclose(o_all, o_n, atol=1e-14) and np.allclose(l_all, l_n, atol=1e-14)
    # a single part is returned unchanged; all-empty gives O = 0, lse = -inf
    o1, l1 = att.lse_combine(o[:1], l[:1])
    assert np.allclose(o1, o[0]) and np.allclose(l1, l[0])
    oe, le = att.lse_combine(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(oe == 0) and np.all(np.isneginf(le))
    # weights are softmax(lse): compare with scipy
    w = np.exp(l - logsumexp(l, axis=0))
    assert np.allclose(o_all, np.einsum("pr,prd->rd", w, o), atol=1e-14)
    assert np.allclose(l_all, logsumexp(l, axis=0), atol=1e-14)


def test_fanout_reference_equals_prefix_suffix_split():
    rng = np.random.default_rng(8)
    a_n, hq, hkv, d, p, s = 3, 4, 2, 32, 40, 9
    q16 = rng.standard_normal((a_n, hq, d)).astype(np.float16)
    pk = rng.standard_normal((p, hkv, d)).astype(np.float16)
    pv = rng.standard_normal((p, hkv, d)).astype(np.float16)
    sk = rng.standard_normal((a_n, s, hkv, d)).astype(np.float16)
    sv = rng.standard_normal((a_n, s, hkv, d)).astype(np.float16)
    words = np.array([0x12345678], dtype=np.int64)
    o, l = pipeline.fanout_reference(q16, pk, pv, sk, sv, "q8_0", "tq3", 0.2, 0.0, words)
    kp = pipeline.dequant("q8_0", pk)
    vp = pipeline.dequant("tq3", pv, words)
    pre = att.gqa_decode(q16.astype(np.float64), kp, vp, 0.2)
    for a in range(a_n):
        suf = att.gqa_decode(q16[a:a + 1].astype(np.float64), sk[a].astype(np.float64),
                             sv[a].astype(np.float64), 0.2)
        oc, lc = att.lse_combine(np.stack([pre[0][a:a + 1], suf[0]]), np.stack([pre[1][a:a + 1], suf[1]]))
        assert np.allclose(oc[0], o[a], atol=1e-13) and np.allclose(lc[0], l[a], atol=1e-13)


def _mixed_inputs(seed, n=37, hq=4, hkv=2, d=32):
    rng = np.random.default_rng(seed)
    q16 = (rng.standard_normal((1, hq, d)) * 2).astype(np.float16)
    k16 = rng.standard_normal((n, hkv, d)).astype(np.float16)
    v16 = rng.standard_normal((n, hkv, d)).astype(np.float16)
    return q16, k16, v16, np.array([0x9E3779B9], dtype=np.int64)


def test_mixed_reference_reduces_to_uniform():
    """Tail formats equal to the window's, and the two extreme window lengths, give
    exactly the uniform-format reference."""
    q16, k16, v16, w = _mixed_inputs(11)
    n = k16.shape[0]
    ref = pipeline.layer_reference(q16, k16, v16, "q8_0", "tq3", 0.25, 0.0, w)
    for wc in (0, 13, n):
        o, l = pipeline.mixed_layer_reference(q16, k16, v16, wc, "q8_0", "tq3", "q8_0", "tq3", 0.25, 0.0, w)
        assert np.array_equal(o, ref[0]) and np.array_equal(l, ref[1]), wc
    tail_only = pipeline.layer_reference(q16, k16, v16, "f16", "q8_0", 0.25, 0.0, w)
    o, l = pipeline.mixed_layer_reference(q16, k16, v16, 0, "q8_0", "tq3", "f16", "q8_0", 0.25, 0.0, w)
    assert np.array_equal(o, tail_only[0]) and np.array_equal(l, tail_only[1])
    window_only = pipeline.layer_reference(q16, k16, v16, "q8_0", "tq3", 0.25, 0.0, w)
    o, l = pipeline.mixed_layer_reference(q16, k16, v16, n, "q8_0", "tq3", "f16", "q8_0", 0.25, 0.0, w)
    assert np.array_equal(o, window_only[0]) and np.array_equal(l, window_only[1])


@pytest.mark.parametrize("wc", [1, 16, 36])
def test_mixed_reference_brute_force_per_position(wc):
    """Each position read at the format of its own range, checked by explicit loops
    (a swapped range or an off-by-one at wc changes the result)."""
    q16, k16, v16, w = _mixed_inputs(12 + wc)
    n, hkv = k16.shape[0], k16.shape[1]
    hq = q16.shape[1]
    o, l = pipeline.mixed_layer_reference(q16, k16, v16, wc, "f16", "f16", "q8_0", "tq3", 0.3, 2.0, w)
    for h in range(hq):
        g = h // (hq // hkv)
        ks, vs = [], []
        for t in range(n):
            kf, vf = ("f16", "f16") if t < wc else ("q8_0", "tq3")
            ks.append(pipeline.dequant(kf, k16[t:t + 1, g], w)[0])
            vs.append(pipeline.dequant(vf, v16[t:t + 1, g], w)[0])
        ob, lb = att.attend_loops(q16[0, h:h + 1].astype(np.float64), np.array(ks), np.array(vs), 0.3, 2.0)
        assert np.allclose(o[0, h], ob[0], atol=1e-12) and abs(l[0, h] - lb[0]) < 1e-12
    # and the tail really is read at its own format: with the tail at fp16 the output moves
    o2, _ = pipeline.mixed_layer_reference(q16, k16, v16, wc, "f16", "f16", "f16", "f16", 0.3, 2.0, w)
    assert not np.allclose(o, o2, atol=1e-6)


def test_mixed_reference_is_the_combine_of_its_two_parts():
    """The position-split method: window part at the window formats, tail part at the
    tail formats, merged by the LSE combine, equals the mixed reference."""
    q16, k16, v16, w = _mixed_inputs(21)
    wc = 19
    o, l = pipeline.mixed_layer_reference(q16, k16, v16, wc, "q8_0", "q8_0", "q8_0", "tq3", 0.2, 0.0, w)
    q = q16.astype(np.float64)
    pw = att.gqa_decode(q, pipeline.dequant("q8_0", k16[:wc]), pipeline.dequant("q8_0", v16[:wc]), 0.2)
    pt = att.gqa_decode(q, pipeline.dequant("q8_0", k16[wc:]), pipeline.dequant("tq3", v16[wc:], w), 0.2)
    oc, lc = att.lse_combine(np.stack([pw[0], pt[0]]), np.stack([pw[1], pt[1]]))
    assert np.allclose(oc, o, atol=1e-13) and np.allclose(lc, l, atol=1e-13)


def _mq_inputs(seed, n_q=4, n=29, hq=6, hkv=2, d=16):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n_q, hq, d)) * 1.5, rng.standard_normal((n, hkv, d)),
            rng.standard_normal((n, hkv, d)))


def test_multi_query_single_token_and_no_limit_reduce_to_decode():
    q, k, v = _mq_inputs(31)
    o, l = att.multi_query_decode(q[:1], k, v, 0.4)
    r = att.gqa_decode(q[:1], k, v, 0.4)
    assert np.array_equal(o, r[0]) and np.array_equal(l, r[1])
    # a causal limit at or past the end changes nothing
    o1, l1 = att.multi_query_decode(q, k, v, 0.4, 1.0)
    o2, l2 = att.multi_query_decode(q, k, v, 0.4, 1.0, q_pos=k.shape[0] - 1)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("q_pos,begin,end", [(20, 0, 29), (3, 0, 29), (10, 5, 25), (-2, 0, 29)])
def test_multi_query_causal_matches_sdpa_mask_and_loops(q_pos, begin, end):
    """Query token i sees positions p in [begin, end) with p <= q_pos + i: checked
    against torch SDPA with an explicit boolean mask (float64) and against loops."""
    q, k, v = _mq_inputs(32 + q_pos)
    n_q, hq = q.shape[0], q.shape[1]
    g = hq // k.shape[1]
    o, l = att.multi_query_decode(q, k, v, 0.35, 0.0, begin, end, q_pos)
    pos = torch.arange(k.shape[0])
    for h in range(hq):
        kk = torch.from_numpy(k[:, h // g]).double()
        vv = torch.from_numpy(v[:, h // g]).double()
        qq = torch.from_numpy(q[:, h]).double()
        mask = (pos[None, :] >= begin) & (pos[None, :] < end) & (pos[None, :] <= q_pos + torch.arange(n_q)[:, None])
        for i in range(n_q):
            vis = mask[i]
            if not bool(vis.any()):
                assert np.all(o[i, h] == 0) and np.isneginf(l[i, h])
                continue
            ref = torch.nn.functional.scaled_dot_product_attention(qq[i:i + 1][None], kk[None], vv[None],
                                                                   attn_mask=vis[None, None], scale=0.35)[0, 0]
            assert np.allclose(o[i, h], ref.numpy(), atol=1e-12)
            s = (qq[i] @ kk[vis].T).numpy() * 0.35
            assert abs(l[i, h] - logsumexp(s)) < 1e-12
            ob, lb = att.attend_loops(q[i:i + 1, h], k[vis.numpy(), h // g], v[vis.numpy(), h // g], 0.35)
            assert np.allclose(o[i, h], ob[0], atol=1e-12) and abs(l[i, h] - lb[0]) < 1e-12


def test_multi_query_causal_split_identity():
    """Position-split with a causal limit: the parts [0, m) and [m, n) each masked by
    the same absolute q_pos, merged, equal the unsplit result for every m."""
    q, k, v = _mq_inputs(40, n_q=5, n=23)
    n = k.shape[0]
    ref = att.multi_query_decode(q, k, v, 0.3, 0.0, q_pos=n - 5)
    for m in range(0, n + 1):
        a = att.multi_query_decode(q, k, v, 0.3, 0.0, 0, m, q_pos=n - 5)
        b = att.multi_query_decode(q, k, v, 0.3, 0.0, m, n, q_pos=n - 5)
        oc, lc = att.lse_combine(np.stack([a[0], b[0]]), np.stack([a[1], b[1]]))
        assert np.allclose(oc, ref[0], atol=1e-13) and np.allclose(lc, ref[1], atol=1e-13), m
