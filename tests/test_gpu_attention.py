"""GPU decode attention, split and combine vs the float64 oracle."""

import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import pipeline
from oracle import turboquant as otq
from tests.helpers import assert_parity, parity_report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qps():
    import quantized_position_split_gb300 as q
    from quantized_position_split_gb300 import build
    build.build()
    return q


def _inputs(n, hq, hkv, d, seed, outliers=True):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((1, hq, d), generator=g).half()
    k = torch.randn((n, hkv, d), generator=g)
    if outliers:
        for h in range(hkv):
            k[:, h, torch.randperm(d, generator=g)[:4]] *= 20
    v = torch.randn((n, hkv, d), generator=g).half()
    return q, k.half(), v


@pytest.mark.parametrize("n_parts,d", [(7, 128), (1, 32), (10, 128), (38, 256), (201, 512), (64, 1024)])
def test_lse_combine(qps, n_parts, d):
    """Part counts that launch one, two, five and eight warps per CTA (one per eight
    parts), eight of them striding over 201 parts, every head_dim slice count, an empty
    part and a row whose parts are all empty."""
    g = torch.Generator().manual_seed(n_parts * 7 + d)
    o = torch.randn((n_parts, 33, d), generator=g)
    l = torch.randn((n_parts, 33), generator=g) * 5
    l[min(2, n_parts - 1), :7] = -float("inf")
    l[:, 5] = -float("inf")  # a row with every part empty
    oo, ll = qps.lse_combine(o.cuda(), l.cuda())
    ro, rl = oatt.lse_combine(o.numpy(), l.numpy())
    assert np.allclose(oo.cpu().numpy(), ro, atol=2e-6)
    assert np.allclose(ll.cpu().numpy()[np.isfinite(rl)], rl[np.isfinite(rl)], atol=2e-6)
    assert np.all(oo.cpu().numpy()[5] == 0) and np.isneginf(ll.cpu().numpy()[5])


FORMATS = [("f16", "f16"), ("q8_0", "q8_0"), ("q8_0", "tq3"), ("f16", "tq3"), ("q8_0", "f16"),
           ("q8_0", "tq2"), ("q8_0", "tq4"), ("f16", "tq2"), ("f16", "tq4")]


def _encode(qps, layout, fmt, x, words):
    if layout == "head":
        return qps.encode_kv_head_major(fmt, x.cuda(), words)
    return qps.encode_kv(fmt, x.cuda(), words)


LAYOUT_PATH = {"head": "tensor-core", "token": "cuda-core"}


@pytest.mark.parametrize("layout", ["head", "token"])
@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("kf,vf", FORMATS)
@pytest.mark.parametrize("softcap", [0.0, 30.0])
def test_window_attention_formats(qps, layout, d, kf, vf, softcap):
    hq, hkv, n = 8, 2, 1000 + 7
    q, k, v = _inputs(n, hq, hkv, d, seed=d + len(kf) * 7 + len(vf), outliers=True)
    words = synth.sign_bits(d, 42)
    K = _encode(qps, layout, kf, k, words)
    V = _encode(qps, layout, vf, v, words)
    qc = q.cuda()
    scale = 1.0 / np.sqrt(d)
    ro, rl = pipeline.layer_reference(q.numpy(), k.numpy(), v.numpy(), kf, vf, scale, softcap, words.numpy())
    for n_split in (0, 1, 5, 4000):  # 4000 > positions: most splits are empty
        a = qps.attn_args(qc, K, V, scale=scale, softcap=softcap, v_signs=words, n_split=n_split)
        assert qps.attn_path(a) == LAYOUT_PATH[layout]
        o, lse = qps.attn_decode_window(a)
        assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(hq, d), rl.reshape(hq),
                      (layout, d, kf, vf, softcap, n_split))


@pytest.mark.parametrize("layout", ["head", "token"])
@pytest.mark.parametrize("d,g", [(512, 128), (256, 128), (128, 64)])
@pytest.mark.parametrize("vf", ["tq2", "tq3", "tq4"])
def test_window_attention_rotation(qps, layout, d, g, vf):
    """A V encoded with the block-diagonal two-sign rotation, read back through the
    attention's inverse transform (its block width and second sign vector)."""
    hq, hkv, n = 8, 2, 700 + 11
    q, k, v = _inputs(n, hq, hkv, d, seed=d + g + len(vf), outliers=True)
    w1, w2 = synth.sign_bits(d, 42), synth.sign_bits(d, 43)
    rot = qps.Rotation(w1, w2, g)
    K = _encode(qps, layout, "q8_0", k, None)
    V = _encode(qps, layout, vf, v, rot)
    kh = pipeline.dequant("q8_0", k.numpy())
    vh = pipeline.dequant(vf, v.numpy(), otq.Rotation(w1.numpy(), w2.numpy(), g))
    ro, rl = oatt.gqa_decode(q.double().numpy(), kh, vh, 1.0 / np.sqrt(d), 30.0)
    for n_split in (0, 3):
        a = qps.attn_args(q.cuda(), K, V, scale=1.0 / np.sqrt(d), softcap=30.0, v_signs=rot, n_split=n_split)
        assert qps.attn_path(a) == LAYOUT_PATH[layout]
        o, lse = qps.attn_decode_window(a)
        assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(hq, d), rl.reshape(hq),
                      (layout, d, g, vf, n_split))
    # the same cache read with the first form's transform is a different (wrong) answer
    a = qps.attn_args(q.cuda(), K, V, scale=1.0 / np.sqrt(d), softcap=30.0, v_signs=w1)
    o, _ = qps.attn_decode_window(a)
    assert np.abs(o.cpu().numpy() - ro.reshape(hq, d)).max() > 1e-2


@pytest.mark.parametrize("layout", ["head", "token"])
@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("tier", ["tq2", "tq3", "tq4"])
@pytest.mark.parametrize("rot", ["first", "block"])
def test_window_attention_turboquant_k(qps, layout, d, tier, rot):
    """K and V in the same TurboQuant tier: K read in the rotated domain against the
    rotated query, with either rotation form, softcap on, several split counts."""
    hq, hkv, n = 8, 2, 900 + 13
    q, k, v = _inputs(n, hq, hkv, d, seed=7 * d + len(tier) + len(rot), outliers=True)
    w1, w2 = synth.sign_bits(d, 42), synth.sign_bits(d, 43)
    g = min(d, 128) if rot == "block" else 0
    lib_rot = qps.Rotation(w1, w2, g) if rot == "block" else w1
    ora_rot = otq.Rotation(w1.numpy(), w2.numpy(), g) if rot == "block" else w1.numpy()
    K = _encode(qps, layout, tier, k, lib_rot)
    V = _encode(qps, layout, tier, v, lib_rot)
    scale = 1.0 / np.sqrt(d)
    ro, rl = pipeline.layer_reference(q.numpy(), k.numpy(), v.numpy(), tier, tier, scale, 30.0, ora_rot)
    for n_split in (0, 1, 6):
        a = qps.attn_args(q.cuda(), K, V, scale=scale, softcap=30.0, v_signs=lib_rot, n_split=n_split)
        assert qps.attn_path(a) == LAYOUT_PATH[layout]
        o, lse = qps.attn_decode_window(a)
        assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(hq, d), rl.reshape(hq),
                      (layout, d, tier, rot, n_split))


def test_turboquant_k_needs_the_same_tier_for_v(qps):
    d, n = 128, 64
    q, k, v = _inputs(n, 4, 1, d, seed=1)
    w = synth.sign_bits(d, 42)
    for kf, vf in [("tq3", "q8_0"), ("tq3", "tq4"), ("tq2", "f16")]:
        a = qps.attn_args(q.cuda(), qps.encode_kv_head_major(kf, k.cuda(), w),
                          qps.encode_kv_head_major(vf, v.cuda(), w), scale=0.1, v_signs=w)
        with pytest.raises(qps.QpsError):
            qps.attn_decode_window(a)


@pytest.mark.parametrize("layout", ["head", "token"])
@pytest.mark.parametrize("begin,end", [(17, 211), (0, 16), (5, 6), (31, 300), (299, 300)])
@pytest.mark.parametrize("d,kf,vf", [(128, "q8_0", "f16"), (512, "q8_0", "tq3"), (64, "q8_0", "tq4"),
                                     (256, "q8_0", "tq2"), (128, "tq4", "tq4"), (512, "tq3", "tq3")])
def test_ragged_ranges(qps, layout, begin, end, d, kf, vf):
    """Sub-ranges whose ends cut 16-token tiles, single tokens and tiny chunks (at
    head_dim 512 several warps share each tile)."""
    hq, hkv, n = 5, 1, 300
    q, k, v = _inputs(n, hq, hkv, d, seed=begin * 7 + end)
    words = synth.sign_bits(d, 5) if vf.startswith("tq") else None
    K = _encode(qps, layout, kf, k, words)
    V = _encode(qps, layout, vf, v, words)
    kh = pipeline.dequant(kf, k.numpy(), None if words is None else words.numpy())
    vh = pipeline.dequant(vf, v.numpy(), None if words is None else words.numpy())
    for n_split in (1, 3):
        a = qps.attn_args(q.cuda(), K, V, scale=0.1, kv_begin=begin, kv_end=end, n_split=n_split, v_signs=words)
        o, lse = qps.attn_decode_window(a)
        ro, rl = oatt.gqa_decode(q.double().numpy(), kh, vh, 0.1, 0.0, begin, end)
        assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(hq, d), rl.reshape(hq),
                      (layout, begin, end, n_split, d))


def test_sub_range_and_empty_range(qps):
    d, hq, hkv, n = 128, 4, 1, 300
    q, k, v = _inputs(n, hq, hkv, d, seed=3)
    K = qps.encode_kv("f16", k.cuda())
    V = qps.encode_kv("f16", v.cuda())
    a = qps.attn_args(q.cuda(), K, V, scale=0.1, kv_begin=17, kv_end=211)
    o, lse = qps.attn_decode_window(a)
    ro, rl = oatt.gqa_decode(q.double().numpy(), k.double().numpy(), v.double().numpy(), 0.1, 0.0, 17, 211)
    assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(hq, d), rl.reshape(hq))
    a = qps.attn_args(q.cuda(), K, V, scale=0.1, kv_begin=50, kv_end=50)
    o, lse = qps.attn_decode_window(a)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_split_identity_every_window_length(qps):
    """Window [0, wc) on device + tail [wc, n) through the ring, merged, equals the
    unsplit oracle for every wc in 0..n."""
    d, hq, hkv, n = 64, 4, 1, 64
    q, k, v = _inputs(n, hq, hkv, d, seed=11, outliers=False)
    ro, rl = oatt.gqa_decode(q.double().numpy(), k.double().numpy(), v.double().numpy(), 0.125)
    K = qps.encode_kv("f16", k.cuda())
    V = qps.encode_kv("f16", v.cuda())
    qc = q.cuda()
    for wc in range(0, n + 1):
        parts = (torch.zeros((64, hq, d), device="cuda"), torch.zeros((64, hq), device="cuda"))
        off = 0
        a = qps.attn_args(qc, K, V, scale=0.125, kv_begin=0, kv_end=wc, n_split=2)
        qps.attn_decode_window(a, parts=parts, part_offset=0)
        off = 2
        tail = [] if wc == n else [(t, min(t + 7, n)) for t in range(wc, n, 7)]
        if tail:
            kh, vh = K.token_slice(wc, n).pinned_copy(), V.token_slice(wc, n).pinned_copy()
            ring = qps.Ring(2, 64 * 1024)
            ring.begin_step([qps.tile_desc(kh, vh, a0 - wc, b0 - wc) for a0, b0 in tail])
            for i in range(len(tail)):
                ta = qps.attn_args(qc, kh, vh, scale=0.125, n_split=1)
                ring.decode_tail(i, ta, parts=parts, part_offset=off)
                off += 1
            ring.end_step()
        o, lse = qps.lse_combine(parts[0][:off], parts[1][:off])
        assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(hq, d), rl.reshape(hq), wc)
        if tail:
            ring.sync()
            ring.close()


@pytest.mark.parametrize("layout", ["head", "token"])
@pytest.mark.parametrize("b", [1, 2, 5])
@pytest.mark.parametrize("kf,vf", [("q8_0", "tq3"), ("q8_0", "tq4"), ("tq3", "tq3")])
def test_gqa_and_shared_batch(qps, layout, b, kf, vf):
    """A shared prefix (batch_stride 0) read by b batch entries (up to 40 query rows
    per KV head) equals each entry attending it alone."""
    d, hq, hkv, n = 128, 16, 2, 777
    g = torch.Generator().manual_seed(5 + b)
    q = torch.randn((b, hq, d), generator=g).half()
    k = torch.randn((n, hkv, d), generator=g).half()
    v = torch.randn((n, hkv, d), generator=g).half()
    words = synth.sign_bits(d, 42)
    K = _encode(qps, layout, kf, k, words)
    V = _encode(qps, layout, vf, v, words)
    a = qps.attn_args(q.cuda(), K, V, scale=0.09, v_signs=words, shared=True)
    o, lse = qps.attn_decode_window(a)
    kh = pipeline.dequant(kf, k.numpy(), words.numpy())
    vh = pipeline.dequant(vf, v.numpy(), words.numpy())
    ro, rl = oatt.gqa_decode(q.double().numpy(), kh, vh, 0.09)
    assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(b * hq, d), rl.reshape(b * hq))


MQ_FORMATS = [(128, "q8_0", "q8_0", 0.0), (128, "f16", "f16", 0.0), (512, "q8_0", "tq3", 50.0),
              (64, "f16", "tq3", 0.0), (256, "q8_0", "f16", 30.0), (128, "q8_0", "tq2", 0.0),
              (256, "q8_0", "tq4", 0.0), (64, "q8_0", "tq4", 30.0), (512, "f16", "tq2", 0.0),
              (128, "tq3", "tq3", 0.0), (512, "tq4", "tq4", 50.0), (64, "tq2", "tq2", 0.0)]


@pytest.mark.parametrize("d,kf,vf,softcap", MQ_FORMATS)
@pytest.mark.parametrize("n_q", [2, 4, 5])
@pytest.mark.parametrize("batch", [1, 2])
def test_multi_query_verify_batch(qps, d, kf, vf, softcap, n_q, batch):
    """n_q query tokens per sequence (verify batch) on the tensor cores, with and
    without the causal limit, several split counts; some causal rows see no position
    of some chunks, and with q_pos below kv_begin the first tokens see none at all."""
    hq, hkv, n = 10 if d <= 128 else 8, 2, 611
    g = torch.Generator().manual_seed(d + 7 * n_q + 31 * batch)
    q = torch.randn((batch, n_q, hq, d), generator=g).half()
    k = torch.randn((batch, n, hkv, d), generator=g).half()
    v = torch.randn((batch, n, hkv, d), generator=g).half()
    words = synth.sign_bits(d, 42)
    K = qps.encode_kv_head_major(kf, k.cuda(), words)
    V = qps.encode_kv_head_major(vf, v.cuda(), words)
    scale = 1.0 / np.sqrt(d)
    for begin, end, q_pos in [(0, n, None), (0, n, n - n_q), (37, 400, 120), (100, 300, 98)]:
        for n_split in (0, 1, 7):
            a = qps.attn_args(q.cuda(), K, V, scale=scale, softcap=softcap, v_signs=words, kv_begin=begin,
                              kv_end=end, n_split=n_split, q_pos=q_pos)
            assert qps.attn_path(a) == "tensor-core"
            o, lse = qps.attn_decode_window(a)
            o, lse = o.cpu().numpy(), lse.cpu().numpy()
            for b in range(batch):
                kh = pipeline.dequant(kf, k[b].numpy(), words.numpy())
                vh = pipeline.dequant(vf, v[b].numpy(), words.numpy())
                ro, rl = oatt.multi_query_decode(q[b].double().numpy(), kh, vh, scale, softcap, begin, end, q_pos)
                rows = slice(b * n_q * hq, (b + 1) * n_q * hq)
                assert_parity(o[rows], lse[rows], ro.reshape(n_q * hq, d), rl.reshape(n_q * hq),
                              (d, kf, vf, n_q, batch, begin, end, q_pos, n_split))


def test_multi_query_paths_that_refuse(qps):
    """Multi-query needs the tensor-core path and per-entry KV."""
    from quantized_position_split_gb300 import _native as N
    d, hq, n = 128, 4, 64
    k = torch.randn((n, 1, d)).half().cuda()
    k2 = torch.randn((n, 2, d)).half().cuda()  # token-major, 2 heads: not token-contiguous
    Kt2 = qps.encode_kv("f16", k2)
    a = qps.attn_args(torch.randn((1, 3, 2, d)).half().cuda(), Kt2, Kt2, scale=0.1)
    assert qps.attn_path(a) == "cuda-core"
    with pytest.raises(N.QpsError) as e:
        qps.attn_decode_window(a)
    assert e.value.status == N.QPS_ERR_UNSUPPORTED
    Kh = qps.encode_kv_head_major("f16", k)
    a = qps.attn_args(torch.randn((2, 3, hq, d)).half().cuda(), Kh, Kh, scale=0.1, shared=True)
    with pytest.raises(N.QpsError) as e:
        qps.attn_plan(a)
    assert e.value.status == N.QPS_ERR_UNSUPPORTED


@pytest.mark.parametrize("pos0,q_pos", [(0, 10), (100, 130), (1000, 1061), (100, 50), (0, None)])
def test_ring_tile_causal_limit_from_its_first_position(qps, pos0, q_pos):
    """A tail tile whose first token sits at view position pos0: a causal q_pos in view
    coordinates limits query token i to the tile positions <= q_pos + i - pos0 (none at
    all when q_pos is before the tile)."""
    d, hq, n, n_q = 128, 4, 64, 3
    g = torch.Generator().manual_seed(pos0 + (q_pos or 0))
    q = torch.randn((1, n_q, hq, d), generator=g).half()
    k = torch.randn((n, 1, d), generator=g).half()
    v = torch.randn((n, 1, d), generator=g).half()
    kh = qps.encode_kv_head_major("f16", k.cuda()).pinned_copy()
    vh = qps.encode_kv_head_major("f16", v.cuda()).pinned_copy()
    ring = qps.Ring(2, 1 << 20)
    ring.begin_step([qps.tile_desc(kh, vh, pos0=pos0)])
    ta = qps.attn_args(q.cuda(), kh, vh, scale=0.1, q_pos=q_pos, n_split=2)
    parts = (torch.zeros((8, n_q * hq, d), device="cuda"), torch.zeros((8, n_q * hq), device="cuda"))
    ring.decode_tail(0, ta, parts=parts, part_offset=0)
    ring.end_step()
    ring.sync()
    ring.close()
    o, lse = qps.lse_combine(parts[0][:2], parts[1][:2])
    ro, rl = oatt.multi_query_decode(q[0].numpy(), k.double().numpy(), v.double().numpy(), 0.1,
                                     q_pos=None if q_pos is None else q_pos - pos0)
    assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(-1, d), rl.reshape(-1), (pos0, q_pos))


def test_zz_no_bounded_wait_gave_up(qps):
    """Every tensor-core launch above finished its tile waits within their bounds."""
    qps.device_status(reset=True)


@pytest.mark.parametrize("flags", [0, 2])
@pytest.mark.parametrize("tokens", [7, 64, 333])
def test_ring_copy_kernel_and_copy_engine_paths(qps, flags, tokens):
    """With the ring's copy kernel selected, a tail tile whose planes live in a
    qps_host_alloc arena is moved by that kernel (one more launch; plane sizes with a
    ragged byte tail), the same tile in torch-pinned memory by cudaMemcpyAsync; both give
    the oracle's answer."""
    d, hq, hkv = 64, 4, 1
    q, k, v = _inputs(tokens, hq, hkv, d, seed=tokens + flags)
    words = synth.sign_bits(d, 42)
    K = qps.encode_kv_head_major("q8_0", k.cuda(), words, pad=1)
    V = qps.encode_kv_head_major("tq3", v.cuda(), words, pad=1)
    kh = pipeline.dequant("q8_0", k.numpy())
    vh = pipeline.dequant("tq3", v.numpy(), words.numpy())
    ro, rl = oatt.gqa_decode(q.double().numpy(), kh, vh, 0.125)
    arena = qps.HostArena(2 << 20, flags)
    launches = []
    for host, mode in (("arena", "kernel"), ("torch", "kernel"), ("arena", "engine")):
        kt = arena.copy_in(K) if host == "arena" else K.pinned_copy()
        vt = arena.copy_in(V) if host == "arena" else V.pinned_copy()
        torch.cuda.synchronize()
        ring = qps.Ring(2, 1 << 20, copy=mode)
        parts = (torch.zeros((4, hq, d), device="cuda"), torch.zeros((4, hq), device="cuda"))
        qps.launch_count(reset=True)
        ring.begin_step([qps.tile_desc(kt, vt)])
        a = qps.attn_args(q.cuda(), kt, vt, scale=0.125, v_signs=words, n_split=1)
        ring.decode_tail(0, a, parts=parts, part_offset=0)
        ring.end_step()
        ring.sync()
        launches.append(qps.launch_count())
        o, lse = qps.lse_combine(parts[0][:1], parts[1][:1])
        assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(hq, d), rl.reshape(hq), (host, mode, flags, tokens))
        ring.close()
    arena.close()
    assert launches[0] == launches[1] + 1  # the arena tile's copy kernel
    assert launches[2] == launches[1]      # the copy engine: no kernel
