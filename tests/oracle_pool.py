"""Oracle layers computed in parallel by spawned CPU worker processes (test
infrastructure only).

Full-size parity compares every layer of a workload with the float64 oracle.  One
oracle layer of the larger workloads costs seconds of single-threaded NumPy, so the
layers are farmed out to a pool of ``spawn``-started processes (never forked: the
parent holds a CUDA context).  Workers import NumPy and ``oracle`` only, each with one
BLAS thread.  Inputs (the fp16 q / K / V the GPU path read, copied to host) are sent
per layer, and at most a few layers are in flight so that the parent never holds more
than that many layers of inputs.
"""

from __future__ import annotations

import concurrent.futures
import multiprocessing
import os

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _mem_available() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 16 << 30


def workers_for(bytes_per_layer: int, cap: int = 0) -> int:
    """Worker count: the host's cores, bounded so that the workers' working sets (at most
    about 10 x one layer's fp16 K + V bytes each: float64 copies of both plus the
    encoders' float32 temporaries) stay within half of the available memory."""
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    by_mem = int(0.5 * _mem_available() // max(1, 10 * bytes_per_layer))
    n = max(1, min(cores, by_mem))
    return min(n, cap) if cap > 0 else n


def _split_layer(job):
    """Worker: expected (O, lse) of one layer of a position-split workload."""
    from oracle import pipeline, turboquant

    (q, k, v, wc, k_fmt, v_fmt, tk_fmt, tv_fmt, scale, softcap, rot) = job
    w1, w2, block = rot
    signs = w1 if w2 is None and block == 0 else turboquant.Rotation(w1, w2, block or None)
    if (tk_fmt, tv_fmt) != (k_fmt, v_fmt):
        return pipeline.mixed_layer_reference(q, k, v, wc, k_fmt, v_fmt, tk_fmt, tv_fmt, scale, softcap, signs)
    return pipeline.layer_reference(q, k, v, k_fmt, v_fmt, scale, softcap, signs)


def split_job(cfg, q, k, v):
    """The picklable job of one layer: host fp16 arrays plus the workload's formats."""
    import synth

    w1, w2, block = synth.rotation_words(cfg)
    rot = (w1.numpy(), None if w2 is None else w2.numpy(), block)
    return (q, k, v, cfg.wc, cfg.k_fmt, cfg.v_fmt, cfg.tk_fmt, cfg.tv_fmt, cfg.scale, cfg.softcap, rot)


class OraclePool:
    """A spawn-context process pool; ``map_bounded`` keeps at most ``inflight`` jobs
    submitted at a time and yields (key, result) as they complete."""

    def __init__(self, workers: int):
        for var in _THREAD_VARS:  # inherited by the spawned workers
            os.environ[var] = "1"
        self.workers = workers
        self.ex = concurrent.futures.ProcessPoolExecutor(max_workers=workers,
                                                         mp_context=multiprocessing.get_context("spawn"))

    def map_bounded(self, fn, jobs, inflight: int = 0):
        """``jobs``: an iterable of (key, job) built lazily; yields (key, fn(job))."""
        inflight = inflight or self.workers + 1
        pending = {}
        it = iter(jobs)
        exhausted = False
        while pending or not exhausted:
            while not exhausted and len(pending) < inflight:
                try:
                    key, job = next(it)
                except StopIteration:
                    exhausted = True
                    break
                pending[self.ex.submit(fn, job)] = key
            if not pending:
                break
            done, _ = concurrent.futures.wait(pending, return_when=concurrent.futures.FIRST_COMPLETED)
            for f in done:
                key = pending.pop(f)
                yield key, f.result()

    def close(self):
        self.ex.shutdown(wait=True, cancel_futures=True)
