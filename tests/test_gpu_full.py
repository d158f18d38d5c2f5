"""Full-size workloads in the configuration the benchmark times (same decoder, same
ring depth and tile size, automatic split counts), checked against the float64 oracle
on EVERY layer, every head and every output element.

The oracle layers run in spawned CPU worker processes (``tests/oracle_pool.py``) while
the decoder's outputs stay on the device; each layer's inputs are drawn again from
their seeded generators on the GPU, exactly as the decoder was loaded.  The step
runner's two degenerate splits run at full size too: no window (wc = 0, every
position streams through the ring) and no tail (wc = n_kv, no ring at all)."""

import pytest
import torch

import synth
from tests import helpers
from tests.helpers import assert_parity
from tests.oracle_pool import OraclePool, _split_layer, split_job, workers_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qps():
    import quantized_position_split_gb300 as q
    from quantized_position_split_gb300 import build
    build.build()
    return q


SPLIT_FULL = ["tiny", "qwen14b_f16", "qwen14b_q8", "gemma_global_q8k_tq3v", "qwen14b_f16_q8tail",
              "qwen14b_q8_tq3vtail", "qwen14b_q8_tq2vtail", "gemma_global_q8k_tq3v_r128",
              "qwen14b_q8_tq3kvtail"]


def check_every_layer(cfg, dec, tag):
    """Compare every layer of ``dec``'s last step with the oracle; returns the worst
    figures seen."""
    per_layer = 2 * max(cfg.n_kv, 1) * cfg.hkv * cfg.d * 2
    pool = OraclePool(workers_for(per_layer, cap=cfg.layers))
    worst = dict(rel_l2=0.0, max_abs=0.0, dlse=0.0)
    seen = set()
    try:
        def jobs():
            for layer in range(cfg.layers):
                q, k, v = helpers.layer_inputs(cfg, layer, "cuda")
                job = split_job(cfg, q[0:cfg.batch].cpu().numpy(), k.cpu().numpy(), v.cpu().numpy())
                del q, k, v
                yield layer, job

        for layer, (ro, rl) in pool.map_bounded(_split_layer, jobs()):
            r = assert_parity(dec.o[layer].cpu().numpy(), dec.lse[layer].cpu().numpy(),
                              ro.reshape(-1, cfg.d), rl.reshape(-1), (tag, layer))
            worst = {key: max(worst[key], r[key]) for key in worst}
            seen.add(layer)
    finally:
        pool.close()
    assert seen == set(range(cfg.layers)), (tag, sorted(set(range(cfg.layers)) - seen))
    return worst


@pytest.mark.parametrize("name", SPLIT_FULL)
def test_full_size_split_workload_every_layer(qps, name):
    cfg = synth.by_name(name)
    dec, _ = helpers.build_split_decoder(cfg)
    dec.step()
    dec.step()  # the second step reuses ring slots whose events belong to step one
    torch.cuda.synchronize()
    qps.device_status(reset=True)
    check_every_layer(cfg, dec, name)
    if dec.ring is not None:
        dec.ring.sync()
    dec.close()


@pytest.mark.parametrize("name,layers", [("qwen14b_f16", 48), ("qwen14b_q8", 4)])
@pytest.mark.parametrize("edge", ["no_window", "no_tail"])
def test_full_size_step_edge_splits(qps, name, layers, edge):
    """qps_decode_step at wc = 0 (tail only: the layers have no device part) and at
    wc = n_kv (window only: no tiles, no ring), full n_kv."""
    base = synth.by_name(name)
    cfg = base.replace(layers=layers, wc=0 if edge == "no_window" else base.n_kv)
    dec, _ = helpers.build_split_decoder(cfg)
    assert (dec.ring is None) == (edge == "no_tail")
    assert dec.n_tiles == (0 if edge == "no_tail" else cfg.layers * len(dec.tile_ranges()))
    for _ in range(2):
        dec.step()
    torch.cuda.synchronize()
    qps.device_status(reset=True)
    check_every_layer(cfg, dec, (name, edge))
    if dec.ring is not None:
        dec.ring.sync()
    dec.close()


def test_full_size_fanout(qps):
    from quantized_position_split_gb300.decode import FanoutDecoder
    cfg = synth.by_name("fanout_prefix")
    ins = helpers.fanout_inputs(cfg, "cuda")
    fd = FanoutDecoder(agents=cfg.agents, hq=cfg.hq, hkv=cfg.hkv, d=cfg.d, k_fmt=cfg.k_fmt,
                       v_fmt=cfg.v_fmt, scale=cfg.scale, softcap=cfg.softcap,
                       signs=helpers.signs_for(cfg)).load(*ins).build()
    fd.step()
    torch.cuda.synchronize()
    ro, rl = helpers.oracle_fanout(cfg, *ins)
    assert_parity(fd.o.cpu().numpy(), fd.lse.cpu().numpy(), ro.reshape(-1, cfg.d), rl.reshape(-1))


def test_zz_no_bounded_wait_gave_up(qps):
    qps.device_status(reset=True)
