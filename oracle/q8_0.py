"""q8_0 block quantisation (oracle).

Source: "F5 M6 — PolyKV (shared compressed KV pool)", section "What PolyKV is
(reference)" (keys kept at int8 / q8_0 because key errors are amplified by the
softmax) and the bits-per-value table of section "S2 tier-family overview" (q8_0 at
1.062 bytes per value).  The numerical definition is the problem statement's: blocks
of 32 consecutive values along head_dim, one fp16 scale d = absmax / 127 per block,
int8 codes.

Readings taken where the pages are silent:
  * the code of x is round(x / d16) where d16 is the STORED fp16 scale (so that the
    round-trip error is at most d16 / 2 whenever d16 is a normal fp16 number; a
    subnormal d16 can round far enough that x / d16 reaches 128 and the clamp costs a
    whole step), rounding half away from zero, clamped to [-127, 127];
  * every step is IEEE float32: d32 = f32(absmax) / 127 (correctly rounded), d16 =
    fp16 round-to-nearest-even of d32, then f32(x) / f32(d16) (correctly rounded);
  * a block whose d16 is zero stores all-zero codes.
"""

from __future__ import annotations

import numpy as np

BLOCK = 32


def encode(x: np.ndarray):
    """Quantise fp16 rows ``x[..., D]`` (D a multiple of 32).

    Returns ``(codes int8 [..., D], scales float16 [..., D // 32])``.
    """
    x = np.asarray(x)
    if x.dtype != np.float16:
        raise TypeError("q8_0 input must be float16")
    d = x.shape[-1]
    if d % BLOCK:
        raise ValueError("head_dim must be a multiple of 32")
    xb = x.astype(np.float32).reshape(x.shape[:-1] + (d // BLOCK, BLOCK))
    amax = np.max(np.abs(xb), axis=-1)  # exact in float32
    d32 = (amax / np.float32(127.0)).astype(np.float32)  # IEEE f32 division
    d16 = d32.astype(np.float16)  # round to nearest even
    dd = d16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (xb / dd).astype(np.float32)  # IEEE f32 division
    # round half away from zero, taken in float64 where |r| + 0.5 is exact
    r64 = ratio.astype(np.float64)
    q = np.sign(r64) * np.floor(np.abs(r64) + 0.5)
    q = np.clip(q, -127, 127)
    q = np.where(dd == 0, 0.0, q)
    codes = q.astype(np.int8).reshape(x.shape)
    return codes, d16


def decode(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantise to float64: x_hat = q * d16, exactly."""
    codes = np.asarray(codes)
    d = codes.shape[-1]
    cb = codes.astype(np.float64).reshape(codes.shape[:-1] + (d // BLOCK, BLOCK))
    out = cb * np.asarray(scales).astype(np.float64)[..., None]
    return out.reshape(codes.shape)


def bytes_per_value(d: int) -> float:
    """Storage per value: one int8 code plus one fp16 scale per 32 values."""
    return (d + 2 * (d // BLOCK)) / d
