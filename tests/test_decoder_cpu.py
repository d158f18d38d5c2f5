"""Host-side planning of the position-split decoder (no GPU): the tail's tiles, the
pinned arena's size and the constructor's argument checks."""

import pytest

from quantized_position_split_gb300 import plane_row_bytes
from quantized_position_split_gb300.decode import PositionSplitDecoder


def _dec(**kw):
    args = dict(layers=3, batch=1, hq=8, hkv=2, d=128, n_kv=1000, wc=333, k_fmt="q8_0", v_fmt="tq3",
                scale=0.1, tile_tokens=200, device="cpu")
    args.update(kw)
    return PositionSplitDecoder(**args)


@pytest.mark.parametrize("n_kv,wc,tile", [(1000, 333, 200), (1000, 0, 1000), (1000, 1000, 64), (17, 5, 4)])
def test_tail_tiles_partition_the_tail(n_kv, wc, tile):
    dec = _dec(n_kv=n_kv, wc=wc, tile_tokens=tile)
    r = dec.tile_ranges()
    covered = [t for a, b in r for t in range(a, b)]
    assert covered == list(range(n_kv - wc))  # every tail position once, in order
    assert all(0 < b - a <= tile for a, b in r)
    assert all(b - a == tile for a, b in r[:-1])  # only the last tile is ragged


@pytest.mark.parametrize("n_kv,wc", [(1000, 333), (1000, 0), (1000, 1000), (17, 16)])
def test_default_tile_is_the_whole_tail_of_a_layer(n_kv, wc):
    args = dict(layers=2, batch=1, hq=8, hkv=2, d=128, n_kv=n_kv, wc=wc, k_fmt="q8_0", v_fmt="q8_0",
                scale=0.1, device="cpu")
    dec = PositionSplitDecoder(**args)  # tile_tokens left at its default
    assert dec.tile_ranges() == ([(0, n_kv - wc)] if n_kv > wc else [])


def test_arena_holds_every_tiles_planes_256_aligned():
    dec = _dec(tail_k_fmt="q8_0", tail_v_fmt="tq2")
    want = 0
    for a, b in dec.tile_ranges():
        tp = -(-(b - a) // 16) * 16  # head-major tile, length padded to 16
        for rb in plane_row_bytes("q8_0", 128) + plane_row_bytes("tq2", 128):
            want += -(-(2 * tp * rb) // 256) * 256
    assert dec._arena_bytes() == 3 * want


def test_constructor_rejects_bad_shapes():
    with pytest.raises(ValueError):
        _dec(wc=1001)
    with pytest.raises(ValueError):
        _dec(n_q=2, batch=2)  # a verify batch decodes one sequence
    with pytest.raises(ValueError):
        _dec(n_q=65)
    dec = _dec(n_q=4)
    assert dec.q.shape == (3, 1, 4, 8, 128) and dec.rows == 32 and dec.q_pos == 996
    assert _dec(n_q=4, causal=False).q_pos is None
