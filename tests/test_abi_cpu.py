"""The C-ABI library without a GPU: it loads, exports every declared symbol, its
struct layouts match the header, and host-side validation rejects bad arguments
before touching the device."""

import ctypes
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

from oracle import turboquant as tq
from quantized_position_split_gb300 import _native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qps.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(N.LIB_PATH):
        from quantized_position_split_gb300 import build
        build.build()
    return N.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^QPS_API\s+[\w\s\*]+?\b(qps_\w+)\(", text, flags=re.M)


def test_header_declares_expected_calls():
    names = set(declared_functions())
    for want in ["qps_kv_quant_q8_0", "qps_kv_quant_tq3", "qps_attn_decode_window",
                 "qps_attn_decode_tail", "qps_lse_combine", "qps_ring_create",
                 "qps_ring_begin_step", "qps_ring_end_step", "qps_decode_step"]:
        assert want in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = declared_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(lib, name), name  # dlsym succeeds
    bound = {s[0] for s in N.SIGNATURES}
    assert set(names) == bound


def test_abi_version_and_status_names(lib):
    m = re.search(r"#define QPS_ABI_VERSION (\d+)", open(HEADER).read())
    assert lib.qps_abi_version() == int(m.group(1))
    assert lib.qps_status_name(0) == b"QPS_OK"
    assert lib.qps_status_name(4) == b"QPS_ERR_TIMEOUT"


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_tier_codebooks_equal_oracle_bit_for_bit(lib, bits):
    n = 1 << bits
    lv = (ctypes.c_float * n)()
    th = (ctypes.c_float * (n - 1))()
    assert lib.qps_tq_codebook(bits, lv, th) == 0
    levels, thresholds = tq.codebook(n)
    assert np.array_equal(np.array(list(lv), dtype=np.float32), levels)
    assert np.array_equal(np.array(list(th), dtype=np.float32), thresholds)
    assert lib.qps_tq_codebook(5, lv, th) == N.QPS_ERR_UNSUPPORTED


def test_codebook_equals_oracle_bit_for_bit(lib):
    lv = (ctypes.c_float * 8)()
    th = (ctypes.c_float * 7)()
    assert lib.qps_tq3_codebook(lv, th) == 0
    levels, thresholds = tq.codebook()
    assert np.array_equal(np.array(list(lv), dtype=np.float32), levels)
    assert np.array_equal(np.array(list(th), dtype=np.float32), thresholds)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "qps.h"\n'
        "int main(void){\n"
        'printf("%zu %zu %zu %zu\\n", sizeof(qps_attn_args), sizeof(qps_tile_desc), sizeof(qps_layer_step), sizeof(qps_kv_view));\n'
        'printf("%zu %zu %zu %zu\\n", offsetof(qps_attn_args, v), offsetof(qps_attn_args, v_signs), offsetof(qps_attn_args, workspace_bytes), offsetof(qps_tile_desc, tokens));\n'
        "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    got = [ctypes.sizeof(N.AttnArgs), ctypes.sizeof(N.TileDesc), ctypes.sizeof(N.LayerStep),
           ctypes.sizeof(N.KvView), N.AttnArgs.v.offset, N.AttnArgs.v_signs.offset,
           N.AttnArgs.workspace_bytes.offset, N.TileDesc.tokens.offset]
    assert [int(x) for x in out] == got


def _args(**kw):
    a = N.AttnArgs()
    a.q = 4096
    a.q_batch_stride = 0
    a.batch, a.hq, a.hkv, a.d = 1, 8, 2, 128
    for side in (a.k, a.v):
        side.fmt = N.FMT_F16
        side.data = 8192
        side.tok_stride = 2
        side.head_stride = 1
        side.batch_stride = 0
    a.kv_begin, a.kv_end = 0, 1000
    a.scale = 0.1
    a.n_split = 4
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_attn_plan_host_only(lib):
    a = _args()
    n = ctypes.c_int32()
    ws = ctypes.c_size_t()
    assert lib.qps_attn_plan(ctypes.byref(a), ctypes.byref(n), ctypes.byref(ws)) == 0
    assert n.value == 4
    assert ws.value >= 4 * 8 * 129 * 4 and ws.value % 256 == 0


@pytest.mark.parametrize("field,value,status", [
    ("hkv", 3, N.QPS_ERR_INVALID_ARG),       # hq not a multiple of hkv
    ("d", 96, N.QPS_ERR_UNSUPPORTED),
    ("kv_end", -1, N.QPS_ERR_INVALID_ARG),
    ("kv_end", 2 ** 31, N.QPS_ERR_UNSUPPORTED),  # beyond 32-bit token coordinates
    ("n_split", -2, N.QPS_ERR_INVALID_ARG),
    ("q", 4098, N.QPS_ERR_INVALID_ARG),      # misaligned
    ("q", None, N.QPS_ERR_INVALID_ARG),
])
def test_attn_validation(lib, field, value, status):
    a = _args(**{field: value})
    assert lib.qps_attn_plan(ctypes.byref(a), None, None) == status
    assert lib.qps_last_error()


def test_attn_view_validation(lib):
    a = _args()
    a.k.fmt = N.FMT_TQ3  # TQ3 is for V only
    a.k.aux = a.k.aux2 = 8192
    assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_ERR_UNSUPPORTED
    a = _args()
    a.v.fmt = N.FMT_Q8_0  # missing scales plane
    assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_ERR_INVALID_ARG
    a = _args()
    a.v.fmt = N.FMT_TQ3
    a.v.aux = a.v.aux2 = 8192  # no sign words
    assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_ERR_INVALID_ARG
    for fmt in (N.FMT_TQ2, N.FMT_TQ4):
        a = _args()
        a.k.fmt = fmt  # TurboQuant tiers are for V only
        a.k.aux = 8192
        assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_ERR_UNSUPPORTED
        a = _args()
        a.v.fmt = fmt
        a.v.aux = 8192  # norms present, no sign words
        assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_ERR_INVALID_ARG
        a.v.aux = 0  # no norms
        assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_ERR_INVALID_ARG
    for blk in (48, 16, 256):  # not a power of two, below 32, above head_dim 128
        a = _args()
        a.v_block = blk
        assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_ERR_INVALID_ARG
    a = _args()
    a.reserved1 = 1
    assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_ERR_INVALID_ARG
    a = _args()
    a.v_block = 64
    assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_OK
    a = _args()
    a.v.fmt = 5  # unknown format
    assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_ERR_INVALID_ARG
    a = _args()
    a.k.batch_stride = 5  # k per batch, v shared
    assert lib.qps_attn_plan(ctypes.byref(a), None, None) == N.QPS_ERR_INVALID_ARG


def test_encoder_and_combine_validation(lib):
    assert lib.qps_kv_quant_q8_0(None, -1, 128, 128, None, None, None) == N.QPS_ERR_INVALID_ARG
    assert lib.qps_kv_quant_q8_0(None, 4, 48, 48, None, None, None) == N.QPS_ERR_UNSUPPORTED
    assert lib.qps_kv_quant_q8_0(None, 0, 128, 128, None, None, None) == N.QPS_OK  # no-op
    assert lib.qps_kv_quant_tq3(None, 4, 128, 128, None, None, None, None, None) == N.QPS_ERR_INVALID_ARG
    w = (ctypes.c_uint32 * 4)()
    assert lib.qps_kv_quant_tq_rot(5, None, 4, 128, 128, w, None, 0, None, None, None, None) == N.QPS_ERR_UNSUPPORTED
    assert lib.qps_kv_quant_tq_rot(3, None, 4, 128, 128, None, None, 0, None, None, None, None) == N.QPS_ERR_INVALID_ARG
    assert lib.qps_kv_quant_tq_rot(3, None, 0, 128, 128, w, None, 96, None, None, None, None) == N.QPS_ERR_INVALID_ARG
    assert lib.qps_kv_quant_tq_rot(4, None, 0, 128, 128, w, None, 32, None, None, None, None) == N.QPS_OK  # no-op
    for fn in (lib.qps_kv_quant_tq2, lib.qps_kv_quant_tq4):
        assert fn(None, 4, 128, 128, None, None, None, None) == N.QPS_ERR_INVALID_ARG
        assert fn(None, 4, 96, 96, None, None, None, None) == N.QPS_ERR_UNSUPPORTED
    assert lib.qps_lse_combine(None, None, 0, 4, 128, None, None, None) == N.QPS_ERR_INVALID_ARG
    assert lib.qps_lse_combine(None, None, 2, 0, 128, None, None, None) == N.QPS_OK  # no rows


def test_binding_tables_match_the_header():
    """The binding's plane sizes and format / copy-mode numbers are the header's."""
    import quantized_position_split_gb300 as qps
    text = open(HEADER).read()
    for name, val in (("QPS_FMT_TQ2", N.FMT_TQ2), ("QPS_FMT_TQ4", N.FMT_TQ4), ("QPS_FMT_TQ3", N.FMT_TQ3)):
        assert re.search(r"%s = %d\b" % (name, val), text), name
    for name, val in (("QPS_RING_COPY_ENGINE", qps.RING_COPY["engine"]), ("QPS_RING_COPY_KERNEL", qps.RING_COPY["kernel"])):
        assert re.search(r"#define %s %d\b" % (name, val), text), name
    d = 256
    assert qps.plane_row_bytes("tq2", d) == [d // 4, 2] and qps.plane_row_bytes("tq4", d) == [d // 2, 2]
    assert qps.plane_row_bytes("tq3", d) == [d // 4, d // 8, 2] and qps.plane_row_bytes("q8_0", d) == [d, d // 16]
    from oracle import turboquant as tq
    for bits, fmt in ((2, "tq2"), (3, "tq3"), (4, "tq4")):  # the binding's sizes are the oracle's bytes per value
        assert (sum(qps.plane_row_bytes(fmt, d))) / d == tq.bytes_per_value(d, bits)


def test_ring_and_step_state_errors(lib):
    assert lib.qps_ring_end_step(None) == N.QPS_ERR_STATE
    assert lib.qps_ring_sync(None, 10) == N.QPS_ERR_STATE
    assert lib.qps_attn_decode_tail(None, 0, None, None) == N.QPS_ERR_STATE
    assert lib.qps_ring_destroy(None) == N.QPS_OK
    assert lib.qps_ring_set_copy_mode(None, 0) == N.QPS_ERR_STATE
    h = ctypes.c_void_p()
    assert lib.qps_ring_create(5, 1024, 0, ctypes.byref(h)) == N.QPS_ERR_INVALID_ARG
    # a step whose layers announce tiles but no ring is given
    st = (N.LayerStep * 1)()
    st[0].n_tiles = 1
    st[0].tail = ctypes.pointer(_args())
    assert lib.qps_decode_step(None, None, 1, st, 1, None) == N.QPS_ERR_INVALID_ARG
    assert lib.qps_decode_step(None, None, 0, st, 1, None) == N.QPS_ERR_INVALID_ARG  # count mismatch


def test_every_declaration_cites_its_source_and_states_its_errors():
    """Each call's comment names the passage it follows (a source tag or a page title)
    or says it has no counterpart on the pages, and states its errors (or that it
    never fails)."""
    text = open(HEADER).read()
    decls = re.findall(r"(/\*(?:(?!\*/).)*\*/)\s*(?:#define[^\n]*\n\s*)*QPS_API\s+[\w\s\*]+?\b(qps_\w+)\(",
                       text, flags=re.S)
    named = {n for _, n in decls}
    assert named == set(declared_functions()) - {"qps_kv_quant_tq4"}  # shares qps_kv_quant_tq2's comment
    for comment, name in decls:
        cites = re.search(r"\[(RKV|RING|POLY|TSTAR)\b", comment) or "counterpart" in comment or '"F5 M' in comment
        assert cites, name
        assert "Errors" in comment or "Never fails" in comment, name


def test_copy_host_argument_checks(lib):
    """qps_copy_host rejects, before any device call, NULL or misaligned pointers and a
    pair of which not exactly one lies in qps_host_alloc memory; zero bytes is a no-op."""
    a = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(a) + 255) // 256 * 256
    assert lib.qps_copy_host(None, base, 64, None) == N.QPS_ERR_INVALID_ARG
    assert lib.qps_copy_host(base, None, 64, None) == N.QPS_ERR_INVALID_ARG
    assert lib.qps_copy_host(base + 8, base + 1024, 64, None) == N.QPS_ERR_INVALID_ARG  # misaligned
    # neither pointer lies in qps_host_alloc memory (ordinary host memory both)
    assert lib.qps_copy_host(base, base + 1024, 64, None) == N.QPS_ERR_INVALID_ARG
    assert "qps_host_alloc" in lib.qps_last_error().decode()
    assert lib.qps_copy_host(base, base + 1024, 0, None) == N.QPS_OK
