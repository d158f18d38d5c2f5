"""Host-side helpers of bench.py (no GPU): the step-time distribution and the host
CPU description."""

import os

import numpy as np
import pytest

import bench


@pytest.mark.parametrize("n", [1, 2, 5, 30, 31])
def test_step_distribution_matches_numpy_percentiles(n):
    rng = np.random.default_rng(n)
    xs = list(rng.uniform(30.0, 35.0, size=n))
    d = bench.step_distribution(xs)
    assert d["p50_ms"] == pytest.approx(np.median(xs), rel=1e-12)
    assert d["p10_ms"] == pytest.approx(np.percentile(xs, 10), rel=1e-12)
    assert d["p90_ms"] == pytest.approx(np.percentile(xs, 90), rel=1e-12)
    assert d["min_ms"] == min(xs) and d["max_ms"] == max(xs)
    assert d["slow_steps"] == 0


def test_step_distribution_counts_slow_steps_and_rejects_empty():
    d = bench.step_distribution([10.0] * 8 + [12.4, 12.6, 300.0])
    assert d["p50_ms"] == 10.0 and d["slow_steps"] == 2 and d["max_ms"] == 300.0
    with pytest.raises(ValueError):
        bench.step_distribution([])


def test_cpu_model_from_cpuinfo_text():
    x86 = "processor\t: 0\nvendor_id\t: GenuineIntel\nmodel name\t: Intel(R) Xeon(R) Processor @ 2.70GHz\n"
    arm = "processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n"
    assert bench.cpu_model(x86) == "Intel(R) Xeon(R) Processor @ 2.70GHz"
    assert bench.cpu_model(arm) == "Arm Neoverse V2 (CPU part 0xd4f)"
    assert bench.cpu_model("CPU part\t: 0xabc\n") == "CPU part 0xabc"
    assert bench.cpu_model("") == "unknown"
    assert bench.cpu_model() != ""


def test_traffic_file_of_a_mixed_tail_is_its_window_kernels():
    import synth
    names = {c.name: bench.traffic_workload(c, synth.CONFIGS) for c in synth.CONFIGS if c.kind == "split"}
    assert names["qwen14b_f16"] == "qwen14b_f16" and names["qwen14b_q8"] == "qwen14b_q8"
    assert names["qwen14b_f16_q8tail"] == "qwen14b_f16"
    for mixed in ("qwen14b_q8_tq3vtail", "qwen14b_q8_tq2vtail", "qwen14b_q8_tq3kvtail"):
        assert names[mixed] == "qwen14b_q8"
    # another rotation is another kernel: the two-sign block rotation keeps its own name
    assert names["gemma_global_q8k_tq3v_r128"] == "gemma_global_q8k_tq3v_r128"
    for c in synth.CONFIGS:
        if c.kind == "split" and c.mixed:
            w = synth.by_name(names[c.name])
            assert (w.wc, w.hkv, w.d, w.k_fmt, w.v_fmt) == (c.wc, c.hkv, c.d, c.k_fmt, c.v_fmt)


def test_committed_traffic_is_dropped_once_the_kernels_change(tmp_path):
    """A DRAM-traffic figure counts only for the kernel sources it was captured on."""
    import json
    import shutil

    src = os.path.join(bench.ROOT, "quantized_position_split_gb300", "csrc")
    shutil.copytree(src, tmp_path / "quantized_position_split_gb300" / "csrc")
    (tmp_path / "profiles").mkdir()
    rec = {"kernel_source_sha": bench.attention_source_sha(str(tmp_path)), "dram_bytes_per_launch": 123.0}
    (tmp_path / "profiles" / "attn_window_w_traffic.json").write_text(json.dumps(rec))
    assert bench.committed_traffic("w", root=str(tmp_path)) == 123.0
    assert bench.committed_traffic("absent", root=str(tmp_path)) is None
    with open(tmp_path / "quantized_position_split_gb300" / "csrc" / "attn_mma.cuh", "a") as f:
        f.write("// edited\n")
    assert bench.committed_traffic("w", root=str(tmp_path)) is None


def test_both_arms_describe_the_workload_with_the_same_config():
    import synth
    args = bench.parse_args([])
    for name in ("qwen14b_q8", "qwen14b_f16", "gemma_global_q8k_tq3v", "fanout_prefix"):
        cfg = synth.by_name(name)
        assert bench.bench_config(cfg, args) == bench.bench_config(cfg, bench.parse_args(["--impl", "reference"]))
    assert bench.parse_args([]).config == "qwen14b_q8"  # the largest single-GPU workload by default
    w, t = bench.split_kv_bytes(synth.by_name("qwen14b_q8"))
    assert abs(w / 1e9 - 10.27) < 0.01 and abs(t / 1e9 - 3.42) < 0.01  # 48 layers x 8 heads x 272 B


def test_both_arms_time_the_same_cut_of_the_workload():
    import synth
    for argv in ([], ["--layers", "3"], ["--tile-tokens", "4096"], ["--config", "qwen14b_f16", "--layers", "2",
                                                                       "--tile-tokens", "16384"]):
        ours = bench.line_workload(synth, bench.parse_args(argv))
        ref = bench.line_workload(synth, bench.parse_args(argv + ["--impl", "reference"]))
        assert ours == ref
        args = bench.parse_args(argv)
        assert bench.bench_config(ours, args) == bench.bench_config(ref, bench.parse_args(argv + ["--impl", "reference"]))
    cut = bench.line_workload(synth, bench.parse_args(["--layers", "3", "--tile-tokens", "4096"]))
    assert (cut.layers, cut.tile_tokens) == (3, 4096)
    assert bench.line_workload(synth, bench.parse_args([])) == synth.by_name("qwen14b_q8")


def test_oracle_sample_spans_the_stack():
    import synth
    assert bench.oracle_layers_for(synth.by_name("qwen14b_q8"), 0) == [0, 16, 31, 47]
    assert bench.oracle_layers_for(synth.by_name("gemma_global_q8k_tq3v"), 0) == [4]
    assert bench.oracle_layers_for(synth.by_name("tiny"), 0) == [0]
    assert bench.oracle_layers_for(synth.by_name("qwen14b_f16"), 2) == [0, 47]


def test_parity_figures_and_the_bar():
    import numpy as np
    ro = np.ones((3, 8))
    rl = np.array([0.0, 1.0, -np.inf])
    ro[2] = 0.0
    f = bench.parity_figures(ro + 1e-4, rl + 5e-5, ro, rl)
    assert f["max_abs"] == pytest.approx(1e-4) and f["dlse"] == pytest.approx(5e-5)
    assert bench.merge_parity([f])["pass"]
    g = bench.parity_figures(ro, np.array([0.0, 1.0, 0.0]), ro, rl)  # an empty row that is not
    assert g["dlse"] == float("inf") and not bench.merge_parity([f, g])["pass"]


def test_reference_arm_line_carries_the_contract_keys(capsys, monkeypatch):
    """The reference arm (the CPU oracle) on the tiny workload, one step: one JSON line
    with the benchmark's keys, its own cpu_baseline and an e2e entry without copies."""
    import json

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0"]) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["metric"] == bench.METRIC and j["unit"] == bench.UNIT
    assert j["value"] > 0 and j["n_gpus"] == 1 and j["steps"] == 1 and j["higher_is_better"] is True
    assert j["config"]["workload"] == "tiny"
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == j["value"] and cb["cores"] >= 1 and cb["sample"]
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_keeps_its_host_time_bounded(capsys, monkeypatch):
    """With a small budget each step samples fewer of the oracle layers, in turn."""
    import json

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", 1e-6)
    monkeypatch.setattr(bench, "oracle_layers_for", lambda cfg, n: [0, 0, 0])
    assert bench.main(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "0"]) == 0
    j = json.loads([ln for ln in capsys.readouterr().out.splitlines() if ln.strip()][-1])
    assert "each step 1 of the layers [0, 0, 0] in turn" in j["cpu_baseline"]["sample"]
    assert j["value"] > 0 and j["steps"] == 2
