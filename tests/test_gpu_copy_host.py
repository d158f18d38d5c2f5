"""qps_copy_host: SM-load copies between device memory and qps_host_alloc memory (the
bench's end-to-end query upload and output readback), byte for byte in both directions,
including a byte tail and a copy that spans most of an arena."""

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qps():
    import quantized_position_split_gb300 as q
    from quantized_position_split_gb300 import build
    build.build()
    return q


@pytest.mark.parametrize("nbytes", [16, 48, 1000, 4099, 491520, (3 << 20) + 7])
def test_round_trip_is_exact(qps, nbytes):
    arena = qps.HostArena(2 * nbytes + 1024)
    try:
        g = torch.Generator().manual_seed(nbytes)
        src = arena.take((nbytes,), torch.uint8)
        src.copy_(torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g))
        back = arena.take((nbytes,), torch.uint8)
        back.zero_()
        dev = torch.full((nbytes,), 7, dtype=torch.uint8, device="cuda")
        s = torch.cuda.current_stream()
        qps.copy_host(dev, src, s)     # host -> device
        dev2 = dev.clone()
        qps.copy_host(back, dev2, s)   # device -> host
        torch.cuda.synchronize()
        assert torch.equal(dev.cpu(), src)
        assert torch.equal(back, src)
        qps.device_status(reset=True)
    finally:
        arena.close()


def test_typed_tensors_and_argument_errors(qps):
    from quantized_position_split_gb300 import _native as N
    arena = qps.HostArena(1 << 16)
    try:
        h = arena.take((40, 128), torch.float32)
        h.copy_(torch.randn(40, 128))
        d = torch.empty((40, 128), dtype=torch.float32, device="cuda")
        qps.copy_host(d, h)
        torch.cuda.synchronize()
        assert torch.equal(d.cpu(), h)
        # two device tensors, two host tensors, different sizes: refused
        for dst, src in ((d, d.clone()), (h, h.clone())):
            with pytest.raises(N.QpsError):
                qps.copy_host(dst, src)
        with pytest.raises(N.QpsError):
            qps.copy_host(d[:20], h)
        # ordinary (not qps_host_alloc) host memory as the device side is refused
        plain = torch.empty((40, 128), dtype=torch.float32)
        rc = qps.lib().qps_copy_host(plain.data_ptr(), h.data_ptr(), h.numel() * 4, None)
        assert rc == N.QPS_ERR_INVALID_ARG
        # a host span that leaves its allocation is refused by the library
        lib = qps.lib()
        end = arena.ptr + arena.nbytes
        assert lib.qps_copy_host(d.data_ptr(), end - 4096, 8192, None) == N.QPS_ERR_INVALID_ARG
    finally:
        arena.close()
