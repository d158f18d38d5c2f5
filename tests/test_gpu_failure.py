"""Failure detection on the GPU without a fault: a bounded in-kernel wait that runs
out.  The library's self-test kernel waits, with the attention kernels' own bounded
wait, on a barrier that nothing arrives on; it must give up after one second of the
GPU's global timer (the recorded duration pins the bound), leave the timeout in the
device error word for qps_device_status to report, and leave the context usable for
the next decode."""

import time

import pytest
import torch

import synth
from tests.helpers import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qps():
    import quantized_position_split_gb300 as q
    from quantized_position_split_gb300 import build
    build.build()
    return q


def test_bounded_wait_gives_up_and_reports_timeout(qps):
    from quantized_position_split_gb300 import _native as N
    torch.cuda.synchronize()
    qps.device_status(reset=True)  # start from a clear error word
    t0 = time.perf_counter()
    qps.selftest_bounded_wait()
    torch.cuda.synchronize()
    rec = qps.device_wait_record()
    with pytest.raises(N.QpsError) as e:
        qps.device_status(reset=True)  # synchronous: waits for the self-test kernel
    assert e.value.status == N.QPS_ERR_TIMEOUT
    assert rec[0] == 1 and 1.0e9 <= rec[12] < 1.2e9, rec  # the wait ran its full second, no more
    assert time.perf_counter() - t0 < 5.0
    assert qps.device_wait_record() == [0] * 16  # the reset cleared the word and the record
    qps.device_status(reset=True)  # the reset cleared it
    # the context still computes: a small decode against the oracle
    cfg = synth.by_name("tiny").replace(n_kv=700, wc=700)
    q = synth.query_f16(cfg, 0, device="cuda")
    k = synth.kv_f16(cfg, 0, "k", cfg.n_kv, device="cuda")
    v = synth.kv_f16(cfg, 0, "v", cfg.n_kv, device="cuda")
    K, V = qps.encode_kv_head_major("f16", k), qps.encode_kv_head_major("f16", v)
    o, lse = qps.attn_decode_window(qps.attn_args(q, K, V, scale=cfg.scale))
    torch.cuda.synchronize()
    from oracle import attention
    ro, rl = attention.gqa_decode(q.cpu().double().numpy(), k.cpu().double().numpy(),
                                  v.cpu().double().numpy(), cfg.scale)
    assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(-1, cfg.d), rl.reshape(-1))
    qps.device_status(reset=True)
