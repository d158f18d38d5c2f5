"""The bounds-checked build (``libqps_checked.so``, QPS_CHECK_BOUNDS=1): the stand-in for
a memory checker where compute-sanitizer cannot be run.

Every kernel of that build tests each staged or addressed access (tensor-map boxes
and zero-filling copies into a tile stage, the rows of a view, q, the partial and
merged outputs, the ring copy kernel's writes into its slot) against its extent,
skips a failing access and marks the device error word (QPS_ERR_INTERNAL).  The
tensor-core window parity over every format pairing and head_dim, whole decode steps
of three workloads, the ring's fault tests and the host copies run under it in a child
process: they must pass, and no check may fail.  The
checker's own report is exercised by its self-test, which guards a store one past a
small shared array (the store is skipped; no access leaves the array)."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHECKED = os.environ.get("QPS_LIB_VARIANT") == "checked"


@pytest.fixture(scope="module")
def checked_lib():
    from quantized_position_split_gb300 import build
    return build.build(variant="checked")


@pytest.mark.skipif(CHECKED, reason="the parent run starts the checked child run")
def test_parity_suites_pass_under_the_checked_build(checked_lib):
    env = dict(os.environ, QPS_LIB_VARIANT="checked")
    # every format pairing and head_dim of the tensor-core window, the split steps of three
    # workloads (fp16, q8_0, the head_dim-512 q8_0-K / TQ3-V one), the ring under faults,
    # the host copies by the ring's copy kernel
    steps = [f"tests/test_gpu_step.py::test_workload_step_parity[{n}]"
             for n in ("qwen14b_f16", "qwen14b_q8", "gemma_global_q8k_tq3v")]
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_checked.py", "tests/test_gpu_attention.py::test_window_attention_formats",
           *steps, "tests/test_gpu_ring_faults.py", "tests/test_gpu_copy_host.py", "-k", "not token"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = (res.stdout + res.stderr)[-4000:]
    assert res.returncode == 0, tail
    assert " passed" in res.stdout and "failed" not in res.stdout, tail


@pytest.mark.skipif(not CHECKED, reason="runs in the checked child process")
def test_the_child_loaded_the_checked_library():
    import quantized_position_split_gb300 as qps
    assert qps.lib().qps_build_checked() == 1


@pytest.mark.skipif(not CHECKED, reason="runs in the checked child process")
def test_the_checker_reports_a_skipped_access():
    import torch

    import quantized_position_split_gb300 as qps
    from quantized_position_split_gb300 import _native as N
    qps.device_status(reset=True)
    N.check(qps.lib().qps_selftest_bounds_check(torch.cuda.current_stream().cuda_stream))
    with pytest.raises(N.QpsError) as e:
        qps.device_status(reset=True)
    assert e.value.status == N.QPS_ERR_INTERNAL and "bounds check" in str(e.value)
    qps.device_status(reset=True)  # cleared


def test_the_default_library_has_no_checks():
    import quantized_position_split_gb300 as qps
    from quantized_position_split_gb300 import _native as N
    if CHECKED:
        pytest.skip("the checked child process")
    assert qps.lib().qps_build_checked() == 0
    assert qps.lib().qps_selftest_bounds_check(None) == N.QPS_ERR_UNSUPPORTED
