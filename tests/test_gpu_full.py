"""Full-size workloads in the configuration the benchmark times (same decoder, same
ring depth and tile size, automatic split counts), checked against the float64 oracle
on sampled layers (each sampled layer is compared on every head and every output
element)."""

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


@pytest.mark.parametrize("name,sample", [
    ("tiny", (0,)),
    ("qwen14b_f16", (0, 47)),
    ("qwen14b_q8", (13,)),
    ("gemma_global_q8k_tq3v", (4,)),
    ("qwen14b_f16_q8tail", (5,)),
    ("qwen14b_q8_tq3vtail", (40,)),
    ("qwen14b_q8_tq2vtail", (21,)),
    ("gemma_global_q8k_tq3v_r128", (2,)),
    ("qwen14b_q8_tq3kvtail", (33,)),
])
def test_full_size_split_workload(qps, name, sample):
    cfg = synth.by_name(name)
    dec, kept = helpers.build_split_decoder(cfg, keep_inputs=sample)
    dec.step()
    dec.step()
    torch.cuda.synchronize()
    for layer in sample:
        q, k, v = kept[layer]
        ro, rl = helpers.oracle_layer(cfg, q, k, v)
        assert_parity(dec.o[layer].cpu().numpy(), dec.lse[layer].cpu().numpy(),
                      ro.reshape(-1, cfg.d), rl.reshape(-1), (name, layer))
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
