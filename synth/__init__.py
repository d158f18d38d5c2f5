"""Seeded synthetic inputs for position-split quantised-KV decode attention.

This package only draws random numbers and describes workload shapes.  It holds
none of the method's arithmetic (no quantisation, no transform, no attention):
both the CUDA path and the CPU oracle take their inputs from here, and neither
imports the other.

Recipe (the same on every device):
  * q, K, V ~ N(0, 1), drawn in float32 from a torch Philox generator whose seed is
    a hash of (base seed, tensor tag), then rounded to fp16 (round to nearest even).
  * "Outlier channels": for K in the Qwen-like and Gemma-like workloads, 4 channel
    indices per (layer, KV head) are drawn without replacement from the same kind of
    generator; those channels of every token are multiplied by 20 before the fp16
    rounding.
  * The TurboQuant sign diagonal is a seeded draw of D random bits (bit i set means
    s_i = -1); seed 42 by default, the rotation seed the PolyKV page names.
"""

from .configs import CONFIGS, Workload, by_name, parity_scaled
from .gen import (
    seed_for,
    randn_f16,
    outlier_channels,
    kv_f16,
    query_f16,
    rotation_words,
    sign_bits,
)

__all__ = [
    "CONFIGS",
    "Workload",
    "by_name",
    "parity_scaled",
    "seed_for",
    "randn_f16",
    "outlier_channels",
    "kv_f16",
    "query_f16",
    "rotation_words",
    "sign_bits",
]
