"""Whole decode steps (window + ring tail + combine) vs the oracle, ring invariances
and the ring's host-side error paths, at parity-sized copies of every workload (every
layer of each), including the step runner's degenerate splits wc = 0 and wc = n_kv."""

import numpy as np
import pytest
import torch

import synth
from tests import helpers
from tests.helpers import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qps():
    import quantized_position_split_gb300 as q
    from quantized_position_split_gb300 import build
    build.build()
    return q


SPLIT_CONFIGS = [c.name for c in synth.CONFIGS if c.kind == "split"]


@pytest.mark.parametrize("name", SPLIT_CONFIGS)
def test_workload_step_parity(qps, name):
    cfg = synth.parity_scaled(synth.by_name(name))
    dec, kept = helpers.build_split_decoder(cfg, keep_inputs=range(cfg.layers))
    assert dec.n_tiles == cfg.layers * len(dec.tile_ranges()) and len(dec.tile_ranges()) >= 3
    import bench
    assert bench.split_kv_bytes(cfg) == (dec.window_bytes(), dec.tail_bytes())  # the bench's byte counts
    for _ in range(2):  # the second step reuses slots whose events belong to step one
        dec.step()
        torch.cuda.synchronize()
        dec.ring.check_guards()  # nothing wrote outside a slot
        for layer, (q, k, v) in kept.items():
            ro, rl = helpers.oracle_layer(cfg, q, k, v)
            assert_parity(dec.o[layer].cpu().numpy(), dec.lse[layer].cpu().numpy(),
                          ro.reshape(-1, cfg.d), rl.reshape(-1), (name, layer))
    dec.ring.sync()
    dec.close()


@pytest.mark.parametrize("name", SPLIT_CONFIGS)
@pytest.mark.parametrize("edge", ["no_window", "no_tail"])
def test_step_edge_splits(qps, name, edge):
    """The combine identity at the ends of the split ("F5 M7 — Rolling KV:
    position-windowed KV residency", section "Implementation decomposition, refined
    (S1 -> S2 -> S3)", item S2): with wc = 0 every position is a tail tile and no layer
    has a device part; with wc = n_kv there are no tiles and no ring.  Both equal plain
    attention over every position."""
    base = synth.parity_scaled(synth.by_name(name), layers=min(4, synth.by_name(name).layers))
    cfg = base.replace(wc=0 if edge == "no_window" else base.n_kv)
    dec, kept = helpers.build_split_decoder(cfg, keep_inputs=range(cfg.layers))
    assert (dec.ring is None) == (edge == "no_tail")
    if edge == "no_window":
        assert dec.window_plan is None and dec.n_tiles == cfg.layers * len(dec.tile_ranges()) >= cfg.layers * 3
    else:
        assert dec.n_tiles == 0
    for _ in range(2):
        dec.step()
        torch.cuda.synchronize()
        if dec.ring is not None:
            dec.ring.check_guards()
        for layer, (q, k, v) in kept.items():
            ro, rl = helpers.oracle_layer(cfg, q, k, v)
            assert_parity(dec.o[layer].cpu().numpy(), dec.lse[layer].cpu().numpy(),
                          ro.reshape(-1, cfg.d), rl.reshape(-1), (name, edge, layer))
    if dec.ring is not None:
        dec.ring.sync()
    dec.close()


@pytest.mark.parametrize("name", ["qwen14b_q8", "qwen14b_q8_tq3vtail", "gemma_global_q8k_tq3v", "qwen14b_q8_tq3kvtail"])
@pytest.mark.parametrize("n_q", [2, 5])
@pytest.mark.parametrize("causal", [True, False])
def test_verify_batch_through_the_split(qps, name, n_q, causal):
    """A verify batch: n_q query tokens at the cache's last positions (in the host tail)
    through window + ring tail + combine; with the causal limit each tile's first
    position reaches the ring.  Small tiles put the limit inside the last tile."""
    from quantized_position_split_gb300.decode import PositionSplitDecoder
    from oracle import attention as oatt
    from oracle import pipeline
    cfg = synth.parity_scaled(synth.by_name(name), layers=1)
    dec = PositionSplitDecoder(layers=1, batch=1, hq=cfg.hq, hkv=cfg.hkv, d=cfg.d, n_kv=cfg.n_kv, wc=cfg.wc,
                               k_fmt=cfg.k_fmt, v_fmt=cfg.v_fmt, scale=cfg.scale, softcap=cfg.softcap,
                               signs=helpers.signs_for(cfg), ring_slots=3, tile_tokens=448,
                               tail_k_fmt=cfg.tail_k_fmt, tail_v_fmt=cfg.tail_v_fmt, n_q=n_q, causal=causal)
    q4 = synth.randn_f16((1, n_q, cfg.hq, cfg.d), cfg.seed, cfg.name, "verify", n_q, device="cuda")
    k = synth.kv_f16(cfg, 0, "k", cfg.n_kv, device="cuda")
    v = synth.kv_f16(cfg, 0, "v", cfg.n_kv, device="cuda")
    dec.load_layer(0, k, v, q4)
    dec.build()
    for _ in range(2):
        dec.step()
        torch.cuda.synchronize()
        sw = helpers.oracle_signs(cfg)
        kn, vn = k.cpu().numpy(), v.cpu().numpy()
        kh = np.concatenate([pipeline.dequant(cfg.k_fmt, kn[:cfg.wc], sw), pipeline.dequant(cfg.tk_fmt, kn[cfg.wc:], sw)])
        vh = np.concatenate([pipeline.dequant(cfg.v_fmt, vn[:cfg.wc], sw), pipeline.dequant(cfg.tv_fmt, vn[cfg.wc:], sw)])
        ro, rl = oatt.multi_query_decode(q4[0].cpu().numpy(), kh, vh, cfg.scale, cfg.softcap,
                                         q_pos=cfg.n_kv - n_q if causal else None)
        assert_parity(dec.o[0].cpu().numpy(), dec.lse[0].cpu().numpy(), ro.reshape(-1, cfg.d), rl.reshape(-1),
                      (name, n_q, causal))
    dec.ring.sync()
    dec.close()


def test_fanout_parity(qps):
    from quantized_position_split_gb300.decode import FanoutDecoder
    cfg = synth.parity_scaled(synth.by_name("fanout_prefix"))
    ins = helpers.fanout_inputs(cfg, "cuda")
    fd = FanoutDecoder(agents=cfg.agents, hq=cfg.hq, hkv=cfg.hkv, d=cfg.d, k_fmt=cfg.k_fmt,
                       v_fmt=cfg.v_fmt, scale=cfg.scale, softcap=cfg.softcap,
                       signs=helpers.signs_for(cfg)).load(*ins).build()
    fd.step()
    torch.cuda.synchronize()
    ro, rl = helpers.oracle_fanout(cfg, *ins)
    assert_parity(fd.o.cpu().numpy(), fd.lse.cpu().numpy(), ro.reshape(-1, cfg.d), rl.reshape(-1))


@pytest.mark.parametrize("name", ["qwen14b_q8", "gemma_global_q8k_tq3v"])
def test_layer_of_several_device_parts_on_side_streams(qps, name):
    """A layer whose positions are cut into five device parts (ragged, one a single
    position) runs its first part on the step's stream and the other four on the
    library's three side streams (one reused); after the join the combine sees every
    part.  Twice in a row, against the oracle over all positions."""
    from quantized_position_split_gb300.decode import _parts_buffers
    cfg = synth.parity_scaled(synth.by_name(name), layers=1)
    q, k, v = helpers.layer_inputs(cfg, 0, "cuda")
    signs = helpers.signs_for(cfg)
    K = qps.encode_kv_head_major(cfg.k_fmt, k, signs)
    V = qps.encode_kv_head_major(cfg.v_fmt, v, signs)
    n = cfg.n_kv
    cuts = [0, 500, 1201, 1202, 1900, n]
    parts = [qps.attn_args(q, K, V, scale=cfg.scale, softcap=cfg.softcap, v_signs=signs, kv_begin=a, kv_end=b)
             for a, b in zip(cuts[:-1], cuts[1:])]
    cap = sum(qps.attn_plan(a)[0] for a in parts)
    rows = cfg.batch * cfg.hq
    o_parts, lse_parts = _parts_buffers(cap, rows, cfg.d, q.device)
    o = torch.zeros((rows, cfg.d), dtype=torch.float32, device=q.device)
    lse = torch.zeros((rows,), dtype=torch.float32, device=q.device)
    plan = qps.StepPlan([dict(device_parts=parts, tail=None, n_tiles=0, o_parts=o_parts, lse_parts=lse_parts,
                              o=o, lse=lse)])
    ro, rl = helpers.oracle_layer(cfg, q, k, v)
    for _ in range(2):
        o.zero_()
        plan.run()
        torch.cuda.synchronize()
        assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(rows, cfg.d), rl.reshape(rows), name)
    qps.device_status(reset=True)


def test_ring_depth_and_tile_invariance(qps):
    cfg = synth.parity_scaled(synth.by_name("qwen14b_q8"), layers=2)
    outs = {}
    for slots, tile in [(2, 512), (3, 512), (4, 512), (3, 300), (2, 2000)]:
        dec, _ = helpers.build_split_decoder(cfg, ring_slots=slots, tile_tokens=tile)
        dec.step()
        torch.cuda.synchronize()
        outs[(slots, tile)] = (dec.o.cpu().clone(), dec.lse.cpu().clone())
        dec.ring.sync()
        dec.close()
    base = outs[(3, 512)]
    for key in [(2, 512), (4, 512)]:  # same tiles: bit-identical whatever the depth
        assert torch.equal(outs[key][0], base[0]) and torch.equal(outs[key][1], base[1]), key
    for key in [(3, 300), (2, 2000)]:
        # other tiles: the same values up to rounding.  The LSE is fp32 throughout; O
        # differs by the fp16 rounding of the softmax weights P, which depends on each
        # tile's running maximum (relative 2^-12 per weight).
        r = helpers.parity_report(outs[key][0].numpy(), outs[key][1].numpy(),
                                  base[0].double().numpy(), base[1].double().numpy())
        assert r["rel_l2"] < 5e-4 and r["dlse"] < 1e-5, (key, r)


def test_ring_host_side_errors(qps):
    from quantized_position_split_gb300 import _native as N
    d, hkv, hq = 128, 2, 4
    k = torch.randn((600, hkv, d)).half()
    K = qps.encode_kv("f16", k.cuda())
    kh = K.pinned_copy()
    q = torch.randn((1, hq, d)).half().cuda()
    parts = (torch.zeros((16, hq, d), device="cuda"), torch.zeros((16, hq), device="cuda"))
    ring = qps.Ring(2, 200 * 1024)
    tiles = [qps.tile_desc(kh, kh, a, a + 100) for a in (0, 100, 200)]
    ring.begin_step(tiles)
    # a second begin while a step is open
    with pytest.raises(N.QpsError) as e:
        ring.begin_step(tiles)
    assert e.value.status == N.QPS_ERR_STATE
    # out of order
    with pytest.raises(N.QpsError) as e:
        ring.decode_tail(1, qps.attn_args(q, kh, kh, scale=0.1, n_split=1), parts=parts, part_offset=0)
    assert e.value.status == N.QPS_ERR_STATE
    ring.decode_tail(0, qps.attn_args(q, kh, kh, scale=0.1, n_split=1), parts=parts, part_offset=0)
    # closing with unconsumed tiles
    with pytest.raises(N.QpsError) as e:
        ring.end_step()
    assert e.value.status == N.QPS_ERR_STATE
    ring.sync()
    # unpinned (pageable) host planes are refused before any copy
    kp = qps.KV("f16", (k.clone(),), 600, hkv, d, hkv)
    with pytest.raises(N.QpsError) as e:
        ring.begin_step([qps.tile_desc(kp, kp, 0, 100)])
    assert e.value.status == N.QPS_ERR_INVALID_ARG
    # a tile larger than a slot
    with pytest.raises(N.QpsError) as e:
        ring.begin_step([qps.tile_desc(kh, kh, 0, 600)])
    assert e.value.status == N.QPS_ERR_INVALID_ARG
    # the ring still works afterwards
    ring.begin_step(tiles[:1])
    ring.decode_tail(0, qps.attn_args(q, kh, kh, scale=0.1, n_split=1), parts=parts, part_offset=0)
    ring.end_step()
    ring.sync()
    ring.close()
    with pytest.raises(N.QpsError):
        ring.handle = None
        N.check(qps.lib().qps_ring_end_step(None))


def test_zz_no_bounded_wait_gave_up(qps):
    qps.device_status(reset=True)
