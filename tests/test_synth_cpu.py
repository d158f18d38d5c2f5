"""The seeded input recipe (synth): deterministic draws, the outlier channels of K, the
sign words, and the parity-sized copies of the workloads."""

import pytest
import torch

import synth


def test_draws_are_deterministic_and_keyed_by_their_tags():
    cfg = synth.by_name("tiny")
    a = synth.kv_f16(cfg, 0, "k", 300)
    assert a.dtype == torch.float16 and a.shape == (300, cfg.hkv, cfg.d)
    assert torch.equal(a, synth.kv_f16(cfg, 0, "k", 300))
    assert not torch.equal(a, synth.kv_f16(cfg, 1, "k", 300))  # another layer
    assert not torch.equal(a, synth.kv_f16(cfg, 0, "v", 300))  # V is its own draw
    assert torch.equal(synth.query_f16(cfg, 0), synth.query_f16(cfg, 0))
    assert synth.query_f16(cfg, 0).shape == (cfg.batch, cfg.hq, cfg.d)


@pytest.mark.parametrize("name", ["qwen14b_f16", "gemma_global_q8k_tq3v"])
def test_k_carries_four_outlier_channels_per_head_scaled_by_20(name):
    cfg = synth.parity_scaled(synth.by_name(name))
    for layer in (0, 1):
        k = synth.kv_f16(cfg, layer, "k", 4000).double()
        std = k.std(dim=0)  # [hkv, d]: per channel over every token
        for h in range(cfg.hkv):
            hot = torch.nonzero(std[h] > 5.0).flatten().tolist()
            assert len(hot) == cfg.k_outliers == 4
            assert all(15.0 < float(std[h, c]) < 25.0 for c in hot)
            cold = [c for c in range(cfg.d) if c not in hot]
            assert float(std[h, cold].max()) < 1.3 and float(std[h, cold].min()) > 0.8
            assert hot == sorted(synth.outlier_channels(cfg.seed, layer, cfg.hkv, cfg.d, 4)[h].tolist())
        v = synth.kv_f16(cfg, layer, "v", 4000).double()
        assert float(v.std(dim=0).max()) < 1.3  # V has no outliers
    c0 = synth.outlier_channels(cfg.seed, 0, cfg.hkv, cfg.d, 4)
    c1 = synth.outlier_channels(cfg.seed, 1, cfg.hkv, cfg.d, 4)
    assert not torch.equal(c0, c1)  # drawn per layer


@pytest.mark.parametrize("d", [32, 64, 128, 512])
def test_sign_words(d):
    w = synth.sign_bits(d, 42)
    assert w.shape == (d // 32,) and int(w.min()) >= 0 and int(w.max()) < 2 ** 32
    ones = sum(bin(int(x)).count("1") for x in w)
    assert 0.3 * d < ones < 0.7 * d
    assert torch.equal(w, synth.sign_bits(d, 42)) and not torch.equal(w, synth.sign_bits(d, 43))
    with pytest.raises(ValueError):
        synth.sign_bits(48)


@pytest.mark.parametrize("cfg", [c for c in synth.CONFIGS if c.kind == "split"], ids=lambda c: c.name)
def test_parity_sized_copies_keep_the_shape_and_cut_ragged(cfg):
    p = synth.parity_scaled(cfg)
    assert (p.hq, p.hkv, p.d, p.k_fmt, p.v_fmt, p.tk_fmt, p.tv_fmt, p.softcap) == \
        (cfg.hq, cfg.hkv, cfg.d, cfg.k_fmt, cfg.v_fmt, cfg.tk_fmt, cfg.tv_fmt, cfg.softcap)
    assert p.n_kv <= 3100 and 0 < p.wc < p.n_kv
    assert p.wc % 16 and p.n_kv % 16 and (p.n_kv - p.wc) % p.tile_tokens  # ragged window and last tile
    assert (p.n_kv - p.wc) // p.tile_tokens >= 2  # several ring tiles
