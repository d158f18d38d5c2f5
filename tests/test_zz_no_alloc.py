"""The allocation-free merged-output entry point (qps_attn_decode_window_noalloc).

Callers that cannot allocate device memory on their call path (an external pool owns
all device memory, or the path must not risk an allocation's synchronisation) use this
entry point; it keeps the split partials in the library's fixed device scratch.  Its
outputs are checked against the float64 oracle and against the workspace entry point,
on two calls in a row.  This file is collected last so that a stop at the first failure
has already run the rest; it also passes on its own in a fresh process.
"""

import ctypes

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


@pytest.mark.parametrize("name,layout", [("qwen14b_q8", "head"), ("gemma_global_q8k_tq3v", "head"),
                                         ("qwen14b_f16", "token")])
def test_noalloc_matches_workspace_entry_point_twice(qps, name, layout):
    cfg = synth.by_name(name).replace(n_kv=3000 + 37, wc=3000 + 37)
    q = synth.query_f16(cfg, 0, device="cuda")
    k = synth.kv_f16(cfg, 0, "k", cfg.n_kv, device="cuda")
    v = synth.kv_f16(cfg, 0, "v", cfg.n_kv, device="cuda")
    signs = synth.sign_bits(cfg.d, cfg.sign_seed)
    enc = qps.encode_kv_head_major if layout == "head" else qps.encode_kv
    K, V = enc(cfg.k_fmt, k, signs), enc(cfg.v_fmt, v, signs)
    a = qps.attn_args(q, K, V, scale=cfg.scale, softcap=cfg.softcap, v_signs=signs)
    ref_o, ref_l = qps.attn_decode_window(a)  # the existing entry point, with a workspace
    # the float64 oracle over every position (the whole cache is the window here)
    oo, ol = helpers.oracle_layer(cfg, q.cpu(), k.cpu(), v.cpu())
    rows = cfg.batch * cfg.hq
    for _ in range(2):  # two calls in a row share and reuse the same scratch
        o = torch.full((rows, cfg.d), float("nan"), device="cuda")
        lse = torch.full((rows,), float("nan"), device="cuda")
        b = qps.attn_args(q, K, V, scale=cfg.scale, softcap=cfg.softcap, v_signs=signs)
        qps.attn_decode_window_noalloc(b, o, lse)
        torch.cuda.synchronize()
        assert_parity(o.cpu().numpy(), lse.cpu().numpy(), oo.reshape(rows, cfg.d), ol.reshape(rows),
                      (name, layout, "oracle"))
        assert_parity(o.cpu().numpy(), lse.cpu().numpy(), ref_o.double().cpu().numpy(),
                      ref_l.double().cpu().numpy(), (name, layout, "workspace entry point"))


@pytest.mark.parametrize("n_q,causal", [(2, 0), (1, 1)])
def test_noalloc_refuses_multi_query_on_the_cuda_core_path(qps, n_q, causal):
    """Token-major planes go to the CUDA-core kernel, which decodes one query token per
    row without a causal limit: the call must refuse, as the workspace entry point does."""
    from quantized_position_split_gb300 import _native as N
    cfg = synth.by_name("qwen14b_f16").replace(n_kv=1000, wc=1000)
    q = synth.randn_f16((1, n_q, cfg.hq, cfg.d), cfg.seed, cfg.name, "noalloc", device="cuda")
    k = synth.kv_f16(cfg, 0, "k", cfg.n_kv, device="cuda")
    K = qps.encode_kv("f16", k)  # token-major: not token-contiguous per head
    a = qps.attn_args(q, K, K, scale=cfg.scale, q_pos=cfg.n_kv - n_q if causal else None)
    a.n_q, a.causal = n_q, causal
    assert qps.attn_path(a) == "cuda-core"
    rows = n_q * cfg.hq
    o = torch.empty((rows, cfg.d), device="cuda")
    lse = torch.empty((rows,), device="cuda")
    with pytest.raises(N.QpsError) as e:
        qps.attn_decode_window_noalloc(a, o, lse)
    assert e.value.status == N.QPS_ERR_UNSUPPORTED
    with pytest.raises(N.QpsError) as e:
        qps.attn_decode_window(a, o=o, lse=lse)
    assert e.value.status == N.QPS_ERR_UNSUPPORTED


def test_noalloc_rejects_requests_beyond_the_scratch(qps):
    from quantized_position_split_gb300 import _native as N
    cfg = synth.by_name("qwen14b_f16").replace(n_kv=4096, wc=4096)
    q = synth.query_f16(cfg, 0, device="cuda")
    k = synth.kv_f16(cfg, 0, "k", cfg.n_kv, device="cuda")
    K = qps.encode_kv_head_major("f16", k)
    # 65535 splits x 40 rows x 129 floats is far beyond 8 MiB
    a = qps.attn_args(q, K, K, scale=cfg.scale, n_split=65535)
    o = torch.empty((cfg.hq, cfg.d), device="cuda")
    lse = torch.empty((cfg.hq,), device="cuda")
    a.o, a.lse = o.data_ptr(), lse.data_ptr()
    st = qps.lib().qps_attn_decode_window_noalloc(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    assert st == N.QPS_ERR_INVALID_ARG
    assert b"scratch" in qps.lib().qps_last_error()
