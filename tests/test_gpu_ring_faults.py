"""The tail ring under host-side faults, and its slot guards ("Rolling-KV:
step/graph-level tail prefetch (design)", section "The fix: a persistent,
step-spanning tail-prefetch ring": each op waits for its tile's copy_done, a slot is
refilled only after its compute_done).

Every fault here is made on the host (``qps_ring_inject_fault``): a tile copy that
reports failure instead of being issued, or one held back by a host function on the
copy stream.  None faults, traps or hangs the GPU.  After each, the ring must report
the right status and then decode exactly again.  The guard test writes one byte into
the guard region after a slot (memory the ring allocated for exactly that purpose)
and expects ``qps_ring_check_guards`` to name the slot."""

import ctypes

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


@pytest.fixture(scope="module")
def workload(qps):
    """A parity-sized two-layer q8_0 workload: 4 tiles per layer through 3 slots."""
    cfg = synth.parity_scaled(synth.by_name("qwen14b_q8"), layers=2)
    dec, kept = helpers.build_split_decoder(cfg, keep_inputs=range(cfg.layers))
    refs = {layer: helpers.oracle_layer(cfg, *kept[layer]) for layer in kept}
    yield cfg, dec, refs
    dec.ring.sync()
    dec.close()


def _check(cfg, dec, refs, tag):
    torch.cuda.synchronize()
    for layer, (ro, rl) in refs.items():
        assert_parity(dec.o[layer].cpu().numpy(), dec.lse[layer].cpu().numpy(), ro.reshape(-1, cfg.d),
                      rl.reshape(-1), (tag, layer))
    dec.ring.check_guards()


@pytest.mark.parametrize("tile", [0, 2, 4, 7])
def test_a_failed_copy_is_reported_and_the_ring_recovers(qps, workload, tile):
    """tiles 0 / 2 fail inside begin_step (the first n_slots copies), 4 and 7 when a
    consumed tile's slot is refilled (the second in the next layer); the step returns
    QPS_ERR_CUDA and the next one is exact."""
    from quantized_position_split_gb300 import _native as N
    cfg, dec, refs = workload
    assert dec.n_tiles == 8 and dec.ring.n_slots == 3
    dec.step()
    _check(cfg, dec, refs, "before")
    dec.o.zero_()
    dec.ring.inject_fault(tile, "copy_fail")
    with pytest.raises(N.QpsError) as e:
        dec.step()
    assert e.value.status == N.QPS_ERR_CUDA and "injected" in str(e.value)
    dec.ring.sync()
    for _ in range(2):
        dec.step()
        _check(cfg, dec, refs, ("after", tile))
    qps.device_status(reset=True)


def test_a_late_copy_holds_the_step_and_sync_times_out(qps, workload):
    """A tile copy held 400 ms on the host: qps_ring_sync with a 50 ms deadline returns
    QPS_ERR_TIMEOUT (never blocks past it), a longer one succeeds, and the step is
    exact: the tail attention waited for the tile's copy_done."""
    import time

    from quantized_position_split_gb300 import _native as N
    cfg, dec, refs = workload
    dec.ring.sync()
    dec.o.zero_()
    dec.ring.inject_fault(5, "copy_late", delay_ms=400)
    dec.step()
    t0 = time.perf_counter()
    with pytest.raises(N.QpsError) as e:
        dec.ring.sync(timeout_ms=50)
    assert e.value.status == N.QPS_ERR_TIMEOUT and time.perf_counter() - t0 < 0.35
    dec.ring.sync(timeout_ms=10000)
    _check(cfg, dec, refs, "late copy")
    qps.device_status(reset=True)


def test_fault_arguments_are_checked(qps, workload):
    from quantized_position_split_gb300 import _native as N
    _, dec, _ = workload
    for args in [(-1, 1, 0), (0, 7, 0), (0, 2, 6000), (0, 2, -1)]:
        assert qps.lib().qps_ring_inject_fault(dec.ring.handle, *args) == N.QPS_ERR_INVALID_ARG
    dec.ring.inject_fault(3, "copy_fail")
    dec.ring.inject_fault(3, "none")  # disarmed: the next steps run clean
    dec.step()
    dec.ring.sync()


def _cudart():
    """The CUDA runtime already loaded in this process (by the library or torch)."""
    with open("/proc/self/maps") as f:
        for line in f:
            path = line.split()[-1]
            if "libcudart.so" in path:
                return ctypes.CDLL(path)
    raise RuntimeError("no CUDA runtime loaded")


@pytest.mark.parametrize("side", ["after", "before"])
def test_a_write_outside_a_slot_is_caught_by_its_guard(qps, side):
    from quantized_position_split_gb300 import _native as N
    ring = qps.Ring(2, 4096)
    ring.check_guards()  # fresh guards
    data, nbytes = ring.slot(1)
    assert nbytes >= 4096 and data % 256 == 0
    rt = _cudart()
    rt.cudaMemset.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t]
    target = data + nbytes if side == "after" else data - 1  # first byte past the slot / last before it
    assert rt.cudaMemset(ctypes.c_void_p(target), 0x5A, 1) == 0
    torch.cuda.synchronize()
    bad = ctypes.c_int32(-7)
    st = qps.lib().qps_ring_check_guards(ring.handle, 1000, ctypes.byref(bad))
    assert st == N.QPS_ERR_INTERNAL and bad.value == 1
    assert side.encode() in qps.lib().qps_last_error()
    ring.close()
