"""The Python binding's marshalling on CPU: the head-major layout addresses every row,
the argument struct carries the shapes, strides and sign words the header describes,
and ring tile descriptors point at the right host bytes.  fp16 caches need no encoder
kernel, and the path / plan queries are host-only, so none of this touches a GPU."""

import ctypes

import numpy as np
import pytest
import torch

import quantized_position_split_gb300 as qps
from quantized_position_split_gb300 import _native as N


def _x(tokens, hkv, d, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((tokens, hkv, d), generator=g).half()


def _row(kv, plane, t, h, b=0):
    """Row (token t, head h, batch b) of a plane, addressed as the header defines."""
    p = kv.planes[plane]
    flat = p.reshape(-1, p.shape[-1])
    return flat[b * kv.batch_stride + t * kv.tok_stride + h * kv.head_stride]


@pytest.mark.parametrize("tokens", [1, 16, 37])
def test_head_major_layout_addresses_every_row(tokens):
    hkv, d = 3, 64
    x = _x(tokens, hkv, d)
    k = qps.encode_kv_head_major("f16", x)
    tp = (tokens + 15) // 16 * 16
    assert k.planes[0].shape == (hkv, tp, d) and (k.tok_stride, k.head_stride) == (1, tp)
    for t in range(tokens):
        for h in range(hkv):
            assert torch.equal(_row(k, 0, t, h), x[t, h])
    assert not k.planes[0][:, tokens:].any()  # the padding rows are zeros
    tm = qps.encode_kv("f16", x)
    assert (tm.tok_stride, tm.head_stride) == (hkv, 1)
    for t in range(tokens):
        for h in range(hkv):
            assert torch.equal(_row(tm, 0, t, h), x[t, h])


def test_batched_head_major_layout():
    x = torch.stack([_x(20, 2, 64, seed=s) for s in range(3)])
    k = qps.encode_kv_head_major("f16", x)
    assert k.batch_stride == 2 * 32
    for b in range(3):
        for t in (0, 7, 19):
            assert torch.equal(_row(k, 0, t, 1, b), x[b, t, 1])


def test_attn_args_fields_path_and_plan():
    batch, hq, hkv, d, n = 2, 6, 3, 64, 37
    q = torch.zeros((batch, hq, d), dtype=torch.float16)
    kh, vh = qps.encode_kv_head_major("f16", _x(n, hkv, d, 1)), qps.encode_kv_head_major("f16", _x(n, hkv, d, 2))
    a = qps.attn_args(q, kh, vh, scale=0.125, softcap=30.0, n_split=3)
    assert (a.batch, a.hq, a.hkv, a.d, a.n_q, a.kv_begin, a.kv_end) == (batch, hq, hkv, d, 1, 0, n)
    assert a.q_batch_stride == hq * d and a.q == q.data_ptr()
    assert (a.k.tok_stride, a.k.head_stride, a.k.fmt) == (1, 48, N.FMT_BY_NAME["f16"])
    assert a.k.data == kh.planes[0].data_ptr() and a.v.data == vh.planes[0].data_ptr()
    assert abs(a.scale - 0.125) < 1e-7 and abs(a.softcap - 30.0) < 1e-6
    assert qps.attn_path(a) == "tensor-core"
    n_split, ws = qps.attn_plan(a)
    rows = batch * hq
    assert n_split == 3 and ws >= 3 * rows * (d + 1) * 4 and ws % 256 == 0
    kt, vt = qps.encode_kv("f16", _x(n, hkv, d, 1)), qps.encode_kv("f16", _x(n, hkv, d, 2))
    assert qps.attn_path(qps.attn_args(q, kt, vt, scale=0.125, n_split=3)) == "cuda-core"
    s = qps.attn_args(q, kh, vh, scale=0.125, n_split=3, shared=True)
    assert s.k.batch_stride == 0 and s.v.batch_stride == 0


def test_multi_query_args():
    q = torch.zeros((1, 4, 8, 128), dtype=torch.float16)
    kh = qps.encode_kv_head_major("f16", _x(50, 2, 128))
    a = qps.attn_args(q, kh, kh, scale=0.1, q_pos=46, n_split=2)
    assert a.n_q == 4 and a.causal == 1 and a.q_pos == 46 and a.q_batch_stride == 4 * 8 * 128
    n_split, ws = qps.attn_plan(a)
    assert n_split == 2 and ws >= 2 * (4 * 8) * 129 * 4
    with pytest.raises(N.QpsError):
        qps.attn_args(q.transpose(1, 2), kh, kh, scale=0.1)  # not contiguous per batch entry


def test_sign_words_and_rotation_reach_the_struct():
    d = 256
    q = torch.zeros((1, 8, d), dtype=torch.float16)
    k = qps.encode_kv_head_major("f16", _x(16, 2, d))
    w1 = np.arange(d // 32, dtype=np.uint32) * np.uint32(0x9E3779B1)
    w2 = w1 ^ np.uint32(0xFFFFFFFF)
    a = qps.attn_args(q, k, k, scale=0.1, v_signs=w1)
    assert [a.v_signs[i] for i in range(d // 32)] == list(w1) and not a.v_signs2 and a.v_block == 0
    b = qps.attn_args(q, k, k, scale=0.1, v_signs=qps.Rotation(w1, w2, 128))
    assert [b.v_signs2[i] for i in range(d // 32)] == list(w2) and b.v_block == 128


def test_tile_desc_of_a_token_major_slice_points_at_its_bytes():
    hkv, d = 2, 64
    x, y = _x(40, hkv, d, 3), _x(40, hkv, d, 4)
    k, v = qps.encode_kv("f16", x), qps.encode_kv("f16", y)
    td = qps.tile_desc(k, v, 5, 20, pos0=7)
    row = hkv * d * 2
    assert (td.tokens, td.tok_stride, td.head_stride, td.pos0) == (15, hkv, 1, 7)
    assert (td.n_k_planes, td.n_v_planes) == (1, 1)
    assert td.host_k[0] == k.planes[0].data_ptr() + 5 * row and td.bytes_k[0] == 15 * row
    got = np.frombuffer(ctypes.string_at(td.host_v[0], td.bytes_v[0]), dtype=np.float16).reshape(15, hkv, d)
    assert np.array_equal(got, y[5:20].numpy())


def test_tile_desc_of_a_whole_head_major_tile():
    kh, vh = qps.encode_kv_head_major("f16", _x(21, 2, 64)), qps.encode_kv_head_major("f16", _x(21, 2, 64, 5))
    td = qps.tile_desc(kh, vh)
    assert (td.tokens, td.tok_stride, td.head_stride) == (21, 1, 32)
    assert td.bytes_k[0] == kh.nbytes() and td.host_v[0] == vh.planes[0].data_ptr()
    with pytest.raises(N.QpsError):
        qps.tile_desc(kh, qps.encode_kv("f16", _x(21, 2, 64)))  # K and V in different layouts
    with pytest.raises(N.QpsError):
        qps.tile_desc(kh, vh, 0, 5)  # slicing needs a token-major cache
