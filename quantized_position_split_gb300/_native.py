"""ctypes declarations of the C ABI in ``include/qps.h`` (argument marshalling only).

The shared library is built in-tree by ``quantized_position_split_gb300.build``; if it
is missing, loading fails loudly: there is no other implementation to fall back to.
``QPS_LIB_VARIANT=checked`` in the environment loads the bounds-checked variant
(``libqps_checked.so``, same ABI) instead.
"""

from __future__ import annotations

import ctypes
import os
import threading
from ctypes import POINTER, c_char_p, c_double, c_float, c_int32, c_int64, c_size_t, c_uint32, c_void_p

LIB_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib")
LIB_PATHS = {"default": os.path.join(LIB_DIR, "libqps.so"), "checked": os.path.join(LIB_DIR, "libqps_checked.so")}
LIB_PATH = LIB_PATHS["default"]


def variant() -> str:
    """The library variant this process loads: "default", or "checked" (bounds checks
    in every kernel) when QPS_LIB_VARIANT=checked."""
    v = os.environ.get("QPS_LIB_VARIANT", "default") or "default"
    if v not in LIB_PATHS:
        raise ImportError(f"QPS_LIB_VARIANT={v!r}: expected one of {sorted(LIB_PATHS)}")
    return v

QPS_OK = 0
QPS_ERR_INVALID_ARG = 1
QPS_ERR_UNSUPPORTED = 2
QPS_ERR_CUDA = 3
QPS_ERR_TIMEOUT = 4
QPS_ERR_STATE = 5
QPS_ERR_INTERNAL = 6

FMT_F16 = 0
FMT_Q8_0 = 1
FMT_TQ3 = 2
FMT_TQ2 = 3
FMT_TQ4 = 4
FMT_BY_NAME = {"f16": FMT_F16, "q8_0": FMT_Q8_0, "tq3": FMT_TQ3, "tq2": FMT_TQ2, "tq4": FMT_TQ4}


class QpsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_name(status)}: {message}")
        self.status = status


class KvView(ctypes.Structure):
    _fields_ = [
        ("fmt", c_int32),
        ("reserved0", c_int32),
        ("data", c_void_p),
        ("aux", c_void_p),
        ("aux2", c_void_p),
        ("tok_stride", c_int64),
        ("head_stride", c_int64),
        ("batch_stride", c_int64),
    ]


class AttnArgs(ctypes.Structure):
    _fields_ = [
        ("q", c_void_p),
        ("q_batch_stride", c_int64),
        ("batch", c_int32),
        ("hq", c_int32),
        ("hkv", c_int32),
        ("d", c_int32),
        ("k", KvView),
        ("v", KvView),
        ("kv_begin", c_int64),
        ("kv_end", c_int64),
        ("scale", c_float),
        ("softcap", c_float),
        ("v_signs", POINTER(c_uint32)),
        ("n_split", c_int32),
        ("part_offset", c_int32),
        ("o_parts", c_void_p),
        ("lse_parts", c_void_p),
        ("o", c_void_p),
        ("lse", c_void_p),
        ("workspace", c_void_p),
        ("workspace_bytes", c_size_t),
        ("n_q", c_int32),
        ("causal", c_int32),
        ("q_pos", c_int64),
        ("v_signs2", POINTER(c_uint32)),
        ("v_block", c_int32),
        ("reserved1", c_int32),
    ]


class TileDesc(ctypes.Structure):
    _fields_ = [
        ("n_k_planes", c_int32),
        ("n_v_planes", c_int32),
        ("host_k", c_void_p * 3),
        ("bytes_k", c_size_t * 3),
        ("host_v", c_void_p * 3),
        ("bytes_v", c_size_t * 3),
        ("tokens", c_int64),
        ("tok_stride", c_int64),
        ("head_stride", c_int64),
        ("pos0", c_int64),
    ]


class LayerStep(ctypes.Structure):
    _fields_ = [
        ("device_parts", POINTER(AttnArgs)),
        ("n_device_parts", c_int32),
        ("n_tiles", c_int32),
        ("tail", POINTER(AttnArgs)),
        ("o_parts", c_void_p),
        ("lse_parts", c_void_p),
        ("parts_capacity", c_int32),
        ("o", c_void_p),
        ("lse", c_void_p),
        ("part_events", c_void_p * 2),
    ]


# (name, restype, argtypes) of every exported function, in header order.
SIGNATURES = [
    ("qps_abi_version", c_int32, []),
    ("qps_last_error", c_char_p, []),
    ("qps_status_name", c_char_p, [c_int32]),
    ("qps_tq3_codebook", c_int32, [POINTER(c_float), POINTER(c_float)]),
    ("qps_tq_codebook", c_int32, [c_int32, POINTER(c_float), POINTER(c_float)]),
    ("qps_kv_quant_q8_0", c_int32, [c_void_p, c_int64, c_int32, c_int64, c_void_p, c_void_p, c_void_p]),
    ("qps_kv_quant_tq3", c_int32,
     [c_void_p, c_int64, c_int32, c_int64, POINTER(c_uint32), c_void_p, c_void_p, c_void_p, c_void_p]),
    ("qps_kv_quant_tq2", c_int32,
     [c_void_p, c_int64, c_int32, c_int64, POINTER(c_uint32), c_void_p, c_void_p, c_void_p]),
    ("qps_kv_quant_tq4", c_int32,
     [c_void_p, c_int64, c_int32, c_int64, POINTER(c_uint32), c_void_p, c_void_p, c_void_p]),
    ("qps_kv_quant_tq_rot", c_int32,
     [c_int32, c_void_p, c_int64, c_int32, c_int64, POINTER(c_uint32), POINTER(c_uint32), c_int32, c_void_p,
      c_void_p, c_void_p, c_void_p]),
    ("qps_attn_plan", c_int32, [POINTER(AttnArgs), POINTER(c_int32), POINTER(c_size_t)]),
    ("qps_attn_path", c_int32, [POINTER(AttnArgs)]),
    ("qps_attn_decode_window", c_int32, [POINTER(AttnArgs), c_void_p]),
    ("qps_lse_combine", c_int32, [c_void_p, c_void_p, c_int32, c_int64, c_int32, c_void_p, c_void_p, c_void_p]),
    ("qps_host_alloc", c_int32, [c_size_t, c_int32, POINTER(c_void_p)]),
    ("qps_host_free", c_int32, [c_void_p]),
    ("qps_copy_host", c_int32, [c_void_p, c_void_p, c_size_t, c_void_p]),
    ("qps_ring_create", c_int32, [c_int32, c_size_t, c_int32, POINTER(c_void_p)]),
    ("qps_ring_destroy", c_int32, [c_void_p]),
    ("qps_ring_set_copy_mode", c_int32, [c_void_p, c_int32]),
    ("qps_ring_begin_step", c_int32, [c_void_p, POINTER(TileDesc), c_int32, c_void_p]),
    ("qps_attn_decode_tail", c_int32, [c_void_p, c_int32, POINTER(AttnArgs), c_void_p]),
    ("qps_ring_end_step", c_int32, [c_void_p]),
    ("qps_ring_sync", c_int32, [c_void_p, c_int32]),
    ("qps_ring_check_guards", c_int32, [c_void_p, c_int32, POINTER(c_int32)]),
    ("qps_ring_slot", c_int32, [c_void_p, c_int32, POINTER(c_void_p), POINTER(c_size_t)]),
    ("qps_ring_inject_fault", c_int32, [c_void_p, c_int32, c_int32, c_int32]),
    ("qps_decode_step", c_int32, [c_void_p, POINTER(TileDesc), c_int32, POINTER(LayerStep), c_int32, c_void_p]),
    ("qps_attn_decode_window_noalloc", c_int32, [POINTER(AttnArgs), c_void_p]),
    ("qps_device_status", c_int32, [c_int32]),
    ("qps_device_wait_record", c_int32, [POINTER(c_uint32), c_int32]),
    ("qps_selftest_bounded_wait", c_int32, [c_void_p]),
    ("qps_build_checked", c_int32, []),
    ("qps_selftest_bounds_check", c_int32, [c_void_p]),
    ("qps_launch_count", c_int64, [c_int32]),
    ("qps_plan_ring", c_int32, [c_double, c_double, c_double, c_double, POINTER(c_int32), POINTER(c_int32),
                                POINTER(c_double), POINTER(c_double)]),
    ("qps_tail_band", c_int32, [c_double, c_double, c_double, c_double, POINTER(c_double)]),
    ("qps_choose_tier", c_int32, [POINTER(c_double), c_int32, c_double, c_double, POINTER(c_int32)]),
]

_lib = None
_lock = threading.Lock()


def load(path: str = None):
    """Load the shared library (the variant ``variant()`` names) once and declare every
    function's signature."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATHS[variant()]
        if not os.path.exists(path):
            raise ImportError(
                f"CUDA library not built: {path} is missing; run "
                "`python -m quantized_position_split_gb300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(path)
        for name, res, args in SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_name(status: int) -> str:
    try:
        return load().qps_status_name(status).decode()
    except ImportError:
        return f"status {status}"


def check(status: int) -> None:
    if status != QPS_OK:
        msg = load().qps_last_error().decode(errors="replace")
        raise QpsError(status, msg)
