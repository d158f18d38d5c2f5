"""Host-side helpers of bench.py (no GPU): the step-time distribution and the host
CPU description."""

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
