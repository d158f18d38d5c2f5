"""Planted mistakes in the oracle, each of which some pin must catch (CPU only).

Every mutant is one small edit of an oracle function's source: a wrong constant, sign,
index, operand, rounding rule or bound.  The edited source is executed in memory as a
fresh namespace and its functions stand in for the real ones for the duration of one
test; nothing is written to disk and the real oracle is restored afterwards.  The pins
of the named test modules then run against the mutated oracle, and the test passes
only if at least one of them fails.  A mutant that every pin accepted would be a
mistake the pins cannot see.
"""

from __future__ import annotations

import importlib
import inspect
import itertools
import types
import warnings

import numpy as np
import pytest

PINS = {
    "q8": ["tests.test_oracle_q8_0"],
    "att": ["tests.test_oracle_attention", "tests.test_oracle_pipeline"],
    "tq": ["tests.test_oracle_tq3", "tests.test_oracle_codebook", "tests.test_oracle_rotation",
           "tests.test_oracle_tqtiers"],
    "pol": ["tests.test_oracle_policy"],
}


def _param_sets(fn):
    """Every argument combination of a test's parametrize marks ([{}] without marks)."""
    axes = []
    for mark in getattr(fn, "pytestmark", []):
        if mark.name != "parametrize":
            continue
        names = mark.args[0]
        names = [s.strip() for s in names.split(",")] if isinstance(names, str) else list(names)
        combos = []
        for v in mark.args[1]:
            v = getattr(v, "values", v)  # pytest.param(...)
            combos.append(dict(zip(names, v if len(names) > 1 else (v,))))
        axes.append(combos)
    return [dict(kv for d in combo for kv in d.items()) for combo in itertools.product(*axes)] or [{}]


def _pins(module_names):
    for mn in module_names:
        mod = importlib.import_module(mn)
        for name, fn in list(vars(mod).items()):
            if name.startswith("test_") and inspect.isfunction(fn) and fn.__module__ == mn:
                for kw in _param_sets(fn):
                    yield f"{mn.rsplit('.', 1)[1]}::{name}{kw or ''}", fn, kw


def _first_failing_pin(module_names):
    """The first pin that fails (label, exception), or None if all pass."""
    for label, fn, kw in _pins(module_names):
        try:
            with np.errstate(all="ignore"), warnings.catch_warnings():
                warnings.simplefilter("ignore")
                fn(**kw)
        except Exception as e:  # an assertion, or an error the planted mistake causes
            return label, e
    return None


def _plant(monkeypatch, module_name, old, new):
    """Replace the functions (and plain constants) of ``module_name`` by those of its
    source with ``old`` replaced by ``new``; ``old`` must occur exactly once."""
    mod = importlib.import_module(module_name)
    src = inspect.getsource(mod)
    assert src.count(old) == 1, f"{old!r} occurs {src.count(old)} times in {module_name}"
    ns = {"__name__": module_name, "__package__": mod.__package__}
    exec(compile(src.replace(old, new), f"<{module_name}, planted mistake>", "exec"), ns)
    for name, val in list(ns.items()):
        orig = getattr(mod, name, None)
        if inspect.isclass(orig) or isinstance(orig, types.ModuleType):
            ns[name] = orig  # keep class identity (isinstance checks) and imported modules
    for name, val in ns.items():
        if inspect.isfunction(val) and inspect.isfunction(getattr(mod, name, None)):
            monkeypatch.setattr(mod, name, val)
        elif isinstance(val, (int, float)) and not isinstance(val, bool) and hasattr(mod, name):
            monkeypatch.setattr(mod, name, val)


# (id, oracle module, original text, planted text, pins that must catch it)
MUTANTS = [
    # q8_0
    ("q8_divisor_128", "oracle.q8_0", "np.float32(127.0)", "np.float32(128.0)", "q8"),
    ("q8_divides_by_unrounded_scale", "oracle.q8_0", "ratio = (xb / dd)", "ratio = (xb / d32[..., None])", "q8"),
    ("q8_rounds_half_to_even", "oracle.q8_0", "np.floor(np.abs(r64) + 0.5)", "np.round(np.abs(r64))", "q8"),
    ("q8_signed_max_not_absmax", "oracle.q8_0", "np.max(np.abs(xb), axis=-1)", "np.max(xb, axis=-1)", "q8"),
    ("q8_decode_uses_first_block_scale", "oracle.q8_0", "np.asarray(scales).astype(np.float64)[..., None]",
     "np.asarray(scales).astype(np.float64)[..., :1, None]", "q8"),
    ("q8_bytes_one_byte_scale", "oracle.q8_0", "(d + 2 * (d // BLOCK)) / d", "(d + (d // BLOCK)) / d", "q8"),
    # attention, combine, split and the whole-layer references
    ("softcap_without_cap_factor", "oracle.attention", "s = softcap * np.tanh(s / softcap)",
     "s = np.tanh(s / softcap)", "att"),
    ("logit_scale_dropped", "oracle.attention", ".T) * scale", ".T)", "att"),
    ("gqa_interleaved_heads", "oracle.attention", "kv = h // g", "kv = h % hkv", "att"),
    ("lse_base_2", "oracle.attention", "lse = (m + np.log(l))[:, 0]", "lse = (m + np.log2(l))[:, 0]", "att"),
    ("lse_without_max", "oracle.attention", "lse = (m + np.log(l))[:, 0]", "lse = np.log(l)[:, 0]", "att"),
    ("output_not_normalised", "oracle.attention", "o = (p @ np.asarray(v, dtype=np.float64)) / l",
     "o = (p @ np.asarray(v, dtype=np.float64))", "att"),
    ("combine_weight_sign", "oracle.attention", "np.exp(lse_parts - m_safe[None])",
     "np.exp(m_safe[None] - lse_parts)", "att"),
    ("combine_lse_without_max", "oracle.attention", "m_safe + np.log(np.where(den > 0, den, 1.0))",
     "np.log(np.where(den > 0, den, 1.0))", "att"),
    ("combine_empty_part_weighted", "oracle.attention", "np.exp(lse_parts - m_safe[None]), 0.0)",
     "np.exp(lse_parts - m_safe[None]), 1.0)", "att"),
    ("window_end_off_by_one", "oracle.attention", "parts = [gqa_decode(q, k, v, scale, softcap, 0, wc)]",
     "parts = [gqa_decode(q, k, v, scale, softcap, 0, max(wc - 1, 0))]", "att"),
    ("causal_limit_excludes_self", "oracle.attention", "q_pos + i + 1", "q_pos + i", "att"),
    ("mixed_tail_read_at_window_format", "oracle.pipeline", "dequant(tail_k_fmt, k16[wc:], sign_words)",
     "dequant(k_fmt, k16[wc:], sign_words)", "att"),
    ("fanout_reads_agent_0_suffix", "oracle.pipeline", "np.asarray(suffix_k16[a], dtype=np.float64)",
     "np.asarray(suffix_k16[0], dtype=np.float64)", "att"),
    # TurboQuant: codebook, transform, encoder, planes, decoder
    ("lloyd_centroid_sign", "oracle.turboquant", "c_new = (pa - pb) / mass", "c_new = (pb - pa) / mass", "tq"),
    ("codebook_negative_half_unreversed", "oracle.turboquant", "levels = np.concatenate([-pos[::-1], pos])",
     "levels = np.concatenate([-pos, pos])", "tq"),
    ("thresholds_off_midpoint", "oracle.turboquant", "((levels[:-1] + levels[1:]) / np.float32(2.0))",
     "((levels[:-1] + 3 * levels[1:]) / np.float32(4.0))", "tq"),
    ("fwht_difference_sign", "oracle.turboquant", "t = (a - b).astype(dtype)", "t = (b - a).astype(dtype)", "tq"),
    ("fwht_last_stage_missing", "oracle.turboquant", "while h < g:", "while h < g // 2:", "tq"),
    ("sign_bit_order_reversed", "oracle.turboquant", "(w[i // 32] >> (i % 32)) & 1",
     "(w[i // 32] >> (31 - i % 32)) & 1", "tq"),
    ("norm_fold_reads_one_half", "oracle.turboquant", "t = (t[..., :h] + t[..., h:2 * h])",
     "t = (t[..., :h] + t[..., :h])", "tq"),
    ("norm_without_sqrt", "oracle.turboquant", "n = np.sqrt(nsq).astype(np.float32)",
     "n = nsq.astype(np.float32)", "tq"),
    ("encoder_skips_sign_diagonal", "oracle.turboquant",
     "u = fwht((x32 * s1.astype(np.float32)).astype(np.float32), dtype=np.float32, block=g)",
     "u = fwht(x32, dtype=np.float32, block=g)", "tq"),
    ("encoder_kappa_inverted", "oracle.turboquant", "z = ((u * kappa).astype(np.float32)",
     "z = ((u / kappa).astype(np.float32)", "tq"),
    ("ties_go_down", "oracle.turboquant", "k += (z >= t).astype(np.int64)", "k += (z > t).astype(np.int64)", "tq"),
    ("negative_magnitudes_reversed", "oracle.turboquant", "mag = np.where(sign, k - half, half - 1 - k)",
     "mag = np.where(sign, k - half, k)", "tq"),
    ("planes_packed_big_endian", "oracle.turboquant", "out |= v[..., j] << (width * j)",
     "out |= v[..., j] << (width * (per - 1 - j))", "tq"),
    ("tq2_field_sign_low", "oracle.turboquant", "return (pack_bits((sign << 1) | mag, 2),), norms",
     "return (pack_bits((mag << 1) | sign, 2),), norms", "tq"),
    ("decode_scale_missing_head_dim", "oracle.turboquant", "(n / np.sqrt(float(d) * g))",
     "(n / np.sqrt(float(g) * g))", "tq"),
    ("decode_sign_inside_transform", "oracle.turboquant", "* s1 * fwht(ck, dtype=np.float64, block=g)",
     "* fwht(ck * s1, dtype=np.float64, block=g)", "tq"),
    ("decode_second_signs_skipped", "oracle.turboquant", "ck = ck * s2", "ck = ck", "tq"),
    ("tq3_bytes_without_sign_plane", "oracle.turboquant", "3: d // 4 + d // 8", "3: d // 4", "tq"),
    # residency and ring sizing policy
    ("ring_without_safety", "oracle.policy", "* bw_eff_gbs * 1e9 * safety", "* bw_eff_gbs * 1e9", "pol"),
    ("ring_slots_capped_at_3", "oracle.policy", "min(4, max(2,", "min(3, max(2,", "pol"),
    ("ring_tiles_floor", "oracle.policy", "math.ceil(per_layer_tail_bytes / tile_bytes_max)",
     "max(1, math.floor(per_layer_tail_bytes / tile_bytes_max))", "pol"),
    ("t_star_engage_sign", "oracle.policy", "(target_drop * t_resident - c_engage_ms)",
     "(target_drop * t_resident + c_engage_ms)", "pol"),
    ("tail_drop_in_seconds", "oracle.policy", "tail_bytes / (bw_eff_gbs * 1e9) * 1e3) / t_resident",
     "tail_bytes / (bw_eff_gbs * 1e9)) / t_resident", "pol"),
    ("tier_fit_strict", "oracle.policy", "if b <= budget_bytes + t_star:", "if b < budget_bytes + t_star:", "pol"),
    # zero rows and blocks, bounds and masks, empty parts, the references' formats
    ("q8_clamp_allows_minus_128", "oracle.q8_0", "np.clip(q, -127, 127)", "np.clip(q, -128, 127)", "q8"),
    ("q8_zero_block_not_zeroed", "oracle.q8_0", "q = np.where(dd == 0, 0.0, q)", "q = np.where(dd == 0, 1.0, q)", "q8"),
    ("softcap_on_unscaled_logit", "oracle.attention",
     "s = (np.asarray(q, dtype=np.float64) @ np.asarray(k, dtype=np.float64).T) * scale\n"
     "    if softcap > 0:\n        s = softcap * np.tanh(s / softcap)",
     "s = (np.asarray(q, dtype=np.float64) @ np.asarray(k, dtype=np.float64).T)\n"
     "    if softcap > 0:\n        s = softcap * np.tanh(s / softcap)\n    s = s * scale", "att"),
    ("causal_limit_ignores_begin", "oracle.attention", "min(end, max(begin, q_pos + i + 1))",
     "min(end, q_pos + i + 1)", "att"),
    ("all_empty_combine_lse_zero", "oracle.attention", "np.log(np.where(den > 0, den, 1.0)), -np.inf)",
     "np.log(np.where(den > 0, den, 1.0)), 0.0)", "att"),
    ("mixed_v_tail_read_at_window_format", "oracle.pipeline", "dequant(tail_v_fmt, v16[wc:], sign_words)",
     "dequant(v_fmt, v16[wc:], sign_words)", "att"),
    ("fanout_prefix_k_not_dequantised", "oracle.pipeline", "kp = dequant(k_fmt, prefix_k16, sign_words)",
     "kp = np.asarray(prefix_k16, dtype=np.float64)", "att"),
    ("fanout_prefix_v_not_dequantised", "oracle.pipeline", "vp = dequant(v_fmt, prefix_v16, sign_words)",
     "vp = np.asarray(prefix_v16, dtype=np.float64)", "att"),
    ("q8_0_read_without_quantisation", "oracle.pipeline", "return q8_0.decode(*q8_0.encode(x16))",
     "return x16.astype(np.float64)", "att"),
    ("tier_read_without_quantisation", "oracle.pipeline",
     "return turboquant.decode_tier(planes, n, sign_words, d, bits)", "return x16.astype(np.float64)", "att"),
    ("zero_row_stores_sign_one", "oracle.turboquant", "k = np.where(zero, levels // 2 - 1, k)",
     "k = np.where(zero, levels // 2, k)", "tq"),
    ("kappa_without_sqrt", "oracle.turboquant", "kappa = np.sqrt(np.float32(d // g), dtype=np.float32)",
     "kappa = np.float32(d // g)", "tq"),
    ("tq4_magnitude_mask_2bit", "oracle.turboquant", "sign, mag = f >> 3, f & 7", "sign, mag = f >> 3, f & 3", "tq"),
    ("unpack_mask_one_bit_wide", "oracle.turboquant", "mask = (1 << width) - 1", "mask = (1 << width)", "tq"),
    ("lloyd_stops_early", "oracle.turboquant", "tol: float = 1e-14", "tol: float = 1e-3", "tq"),
    ("mse_integral_truncated", "oracle.turboquant", "[[-12.0], np.asarray(thresholds, dtype=np.float64), [12.0]]",
     "[[-3.0], np.asarray(thresholds, dtype=np.float64), [3.0]]", "tq"),
    ("decode_sign_order_swapped", "oracle.turboquant", "return np.where(sign == 1, half + mag, half - 1 - mag)",
     "return np.where(sign == 1, half - 1 - mag, half + mag)", "tq"),
    ("slots_ceil", "oracle.policy", "math.floor(slot_budget_bytes / tile_bytes_max)",
     "math.ceil(slot_budget_bytes / tile_bytes_max)", "pol"),
    ("tile_bytes_floor", "oracle.policy", "tile_bytes = int(math.ceil(per_layer_tail_bytes / tiles))",
     "tile_bytes = int(per_layer_tail_bytes // tiles)", "pol"),
    ("t_star_negative_kept", "oracle.policy", "return max(0.0, t)", "return t", "pol"),
    ("no_tier_fits_takes_first", "oracle.policy", "return len(kv_bytes_per_tier) - 1", "return 0", "pol"),
]


@pytest.mark.parametrize("mid,module,old,new,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, mid, module, old, new, pins):
    _plant(monkeypatch, module, old, new)
    caught = _first_failing_pin(PINS[pins])
    assert caught is not None, f"planted mistake {mid!r} ({old!r} -> {new!r}) passes every pin of {PINS[pins]}"


@pytest.mark.parametrize("module,text,pins", [("oracle.q8_0", "BLOCK = 32", "q8"),
                                              ("oracle.attention", "def attend(", "att"),
                                              ("oracle.turboquant", "LEVELS = 8", "tq"),
                                              ("oracle.policy", "def ring_plan(", "pol")])
def test_harness_control_unchanged_source_passes_every_pin(monkeypatch, module, text, pins):
    """The same machinery with an edit that changes nothing: every pin passes, so a
    caught mutant above is caught by its mistake, not by the harness."""
    _plant(monkeypatch, module, text, text)
    assert _first_failing_pin(PINS[pins]) is None
