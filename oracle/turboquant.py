"""TurboQuant-MSE 3-bit ("TQ3") value quantisation (oracle).

Source: "F5 M6 — PolyKV (shared compressed KV pool)":
  * section "What PolyKV is (reference)": V is quantised by a fast Walsh-Hadamard
    rotation that spreads outlier energy over the dimensions, followed by an MSE-optimal
    Lloyd-Max quantiser;
  * section "S2 — TurboQuant tier family": one rotation + codebook scheme,
    parameterised by bit width;
  * section "Phase-0 fork recon": the 3-bit block stores an fp16 norm, a 2-bit plane
    and a 1-bit plane, and the rotation seed is 42;
  * section "S2 perf-path Level B": the cache is read as centroid x norm in the rotated
    domain, and the output is inverse-rotated once (Parseval keeps dot products);
  * the bits-per-value table of section "S2 tier-family overview" (turbo3 at 0.391
    bytes per value).
The problem statement fixes the remaining steps: per-vector L2 norm, seeded +-1 sign
diagonal, orthonormal FWHT over head_dim, 8-level Lloyd-Max codebook fixed by the build.

Readings taken (each one is a choice the pages leave open):
  * Transform: R = H diag(s) / sqrt(D) with H the unnormalised Sylvester-Hadamard
    matrix over the whole head_dim (one sign vector, shared by every layer and head
    of a given D).  The pages' 128-wide block-diagonal and two-sign variants are not
    used.
  * Normalisation: z = H (s * x) / ||x||, so that ||z||^2 = D and each coordinate has
    unit variance; z is quantised with the Gaussian N(0,1) Lloyd-Max codebook.
  * Codebook: the 8-level Lloyd-Max quantiser of N(0,1), solved in float64, with each
    level then rounded to the nearest fp16 value (so that the levels are exact in the
    half-precision tensor-core operands of the read path); the thresholds are the exact
    midpoints of adjacent rounded levels.  The codebook is symmetric.
  * Code of a coordinate: k = number of thresholds t_m with z >= t_m (ties go up).
    Stored as a sign plane hi = (k >= 4) and a magnitude plane lo = k - 4 if hi else
    3 - k, so level = (+1 if hi else -1) * |c|[lo].
  * Norm: the plain L2 norm (the pages' "corrected norm" is not specified), stored as
    fp16; decode is x_hat = (n16 / D) * s * (H c[k]).
  * Encoder arithmetic is IEEE float32 in a fixed order: squares x_i * x_i, then a
    halving fold (for h = D/2, ..., 1: t[i] += t[i + h]); n = sqrt(t[0]) correctly
    rounded; the FWHT butterflies (a, b) -> (a + b, a - b) over stages h = 1, 2, ...,
    D/2; z_i = u_i / n correctly rounded.  A zero row stores all-zero planes and a zero
    norm.
  * Bit order: element i lives in byte i // 4, bits 2 (i % 4) .. 2 (i % 4) + 1 of the
    2-bit plane and in byte i // 8, bit i % 8 of the 1-bit plane.

The tier ladder of section "S2 — TurboQuant tier family" (one rotation + codebook
scheme at several bit widths) adds a 2-bit and a 4-bit tier with the same transform and
norm; their codebooks are the 4- and 16-level Lloyd-Max quantisers of N(0,1), rounded
and made symmetric the same way.  A level index k of a b-bit tier (L = 2^b levels) is
held as sign = (k >= L/2) and magnitude m = k - L/2 if sign else L/2 - 1 - k.  The
pages fix no storage layout for these two tiers; here each element gets one
sign-magnitude field (sign in the top bit, m below), packed little-endian like the TQ3
magnitude plane:
  * TQ2: a 2-bit plane, field (sign << 1) | m, element i at bits 2 (i % 4) of byte i / 4;
  * TQ4: a 4-bit plane, field (sign << 3) | m, element i at bits 4 (i % 2) of byte i / 2;
each with one fp16 norm per vector (the pages' 4-bit block is 2 bytes per vector larger).

The rotation has a second form, the one the pages' fork runs (sections "S2 perf-path
Level B" and the head_dim-512 note after it: the Walsh-Hadamard transform is
block-diagonal over 128-wide blocks, with a sign vector before and another after it):
R = diag(s2) blockdiag(H_G) diag(s1) / sqrt(G) for a block width G dividing D.  The
first form is G = D with s2 = 1.  A ``Rotation(signs1, signs2, block)`` stands wherever
sign words are accepted.  Encoder order: u = FWHT stages h = 1 .. G/2 of s1 .* x (fp32),
then u = s2 .* u (exact), then z = fp32(fp32(u * kappa) / n) with kappa = the float32
square root of D / G (1 when G = D, which leaves the first form unchanged).  Decode:
x_hat = n * s1 .* blockdiag(H_G) (s2 .* c[k]) / sqrt(D G).
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import ndtr

LEVELS = 8


def _phi(x):
    """Standard normal density."""
    return np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def lloyd_max_gaussian(levels: int = LEVELS, tol: float = 1e-14, max_iter: int = 100000):
    """Lloyd iteration for the MSE-optimal scalar quantiser of N(0, 1), in float64.

    Alternates the two optimality conditions until the levels move by less than
    ``tol``: thresholds at midpoints of adjacent levels, and each level at the
    conditional mean of its cell, (phi(a) - phi(b)) / (Phi(b) - Phi(a)).
    Returns ``(levels [L], thresholds [L - 1])`` in float64, ascending.
    """
    c = np.linspace(-2.0, 2.0, levels)
    for _ in range(max_iter):
        t = 0.5 * (c[:-1] + c[1:])
        a = np.concatenate([[-np.inf], t])
        b = np.concatenate([t, [np.inf]])
        pa = np.where(np.isinf(a), 0.0, _phi(np.where(np.isinf(a), 0.0, a)))
        pb = np.where(np.isinf(b), 0.0, _phi(np.where(np.isinf(b), 0.0, b)))
        mass = ndtr(b) - ndtr(a)
        c_new = (pa - pb) / mass
        if np.max(np.abs(c_new - c)) < tol:
            c = c_new
            break
        c = c_new
    t = 0.5 * (c[:-1] + c[1:])
    return c, t


def gaussian_mse(levels: np.ndarray, thresholds: np.ndarray) -> float:
    """Mean squared error of a scalar quantiser on N(0,1), by numerical integration."""
    edges = np.concatenate([[-12.0], np.asarray(thresholds, dtype=np.float64), [12.0]])
    total = 0.0
    for k, c in enumerate(np.asarray(levels, dtype=np.float64)):
        x = np.linspace(edges[k], edges[k + 1], 200001)
        y = (x - c) ** 2 * _phi(x)
        total += float(np.trapezoid(y, x))
    return total


def codebook(levels: int = LEVELS):
    """The build's fixed codebook of ``levels`` levels (8 for TQ3; 4, 16 for TQ2, TQ4).

    Returns ``(levels float32 [L], thresholds float32 [L - 1])``: Lloyd-Max levels of
    N(0,1) rounded to fp16 (held as float32), made exactly symmetric, and the exact
    midpoints between adjacent levels.
    """
    c, _ = lloyd_max_gaussian(levels)
    pos = np.abs(c[levels // 2:]).astype(np.float16).astype(np.float32)
    levels = np.concatenate([-pos[::-1], pos]).astype(np.float32)
    thresholds = ((levels[:-1] + levels[1:]) / np.float32(2.0)).astype(np.float32)
    return levels, thresholds


class Rotation:
    """The transform's parameters: sign words s1 (D/32 words), optional second sign
    words s2 (None: all +1) and the Hadamard block width (None: head_dim)."""

    def __init__(self, signs1, signs2=None, block=None):
        self.signs1 = signs1
        self.signs2 = signs2
        self.block = block


def _rotation(sign_words, d: int):
    """(s1, s2 or None, G) as float64 sign vectors and the block width."""
    if isinstance(sign_words, Rotation):
        g = d if sign_words.block is None else int(sign_words.block)
        if g < 32 or g > d or d % g or g & (g - 1):
            raise ValueError("block must be a power of two in [32, head_dim]")
        s2 = None if sign_words.signs2 is None else signs_from_words(sign_words.signs2, d)
        return signs_from_words(sign_words.signs1, d), s2, g
    return signs_from_words(sign_words, d), None, d


def signs_from_words(words, d: int) -> np.ndarray:
    """Unpack the sign diagonal: bit i of word i // 32 set means s_i = -1 (float64)."""
    w = [int(x) & 0xFFFFFFFF for x in np.asarray(words).reshape(-1).tolist()]
    s = np.ones(d, dtype=np.float64)
    for i in range(d):
        if (w[i // 32] >> (i % 32)) & 1:
            s[i] = -1.0
    return s


def fwht(x: np.ndarray, dtype=np.float64, block=None) -> np.ndarray:
    """Unnormalised fast Walsh-Hadamard transform over the last axis.

    Stages h = 1, 2, 4, ..., D/2; at each stage every pair (i, i + h) with i & h == 0
    becomes (a + b, a - b), each result rounded to ``dtype``.  With ``block`` = G the
    stages stop at G/2: an independent transform of each G-wide block.
    """
    y = np.array(x, dtype=dtype, copy=True)
    d = y.shape[-1]
    if d & (d - 1):
        raise ValueError("length must be a power of two")
    g = d if block is None else block
    lead = y.shape[:-1]
    h = 1
    while h < g:
        z = y.reshape(lead + (d // (2 * h), 2, h))
        a = z[..., 0, :]
        b = z[..., 1, :]
        s = (a + b).astype(dtype)
        t = (a - b).astype(dtype)
        y = np.stack([s, t], axis=-2).reshape(lead + (d,))
        h *= 2
    return y


def _fold_sum_sq_f32(x32: np.ndarray) -> np.ndarray:
    """Sum of squares by a halving fold: for h = D/2 .. 1, t[i] += t[i + h] (float32)."""
    t = (x32 * x32).astype(np.float32)
    d = t.shape[-1]
    h = d // 2
    while h >= 1:
        t = (t[..., :h] + t[..., h:2 * h]).astype(np.float32)
        h //= 2
    return t[..., 0]


def level_index(x: np.ndarray, sign_words, levels: int = LEVELS):
    """Codebook index k [..., D] (0 for a zero row) and fp16 norms of fp16 rows."""
    x = np.asarray(x)
    if x.dtype != np.float16:
        raise TypeError("TurboQuant input must be float16")
    d = x.shape[-1]
    if d % 32 or d & (d - 1):
        raise ValueError("head_dim must be a power of two and a multiple of 32")
    _, thresholds = codebook(levels)
    s1, s2, g = _rotation(sign_words, d)
    x32 = x.astype(np.float32)
    nsq = _fold_sum_sq_f32(x32)
    n = np.sqrt(nsq).astype(np.float32)  # correctly rounded
    u = fwht((x32 * s1.astype(np.float32)).astype(np.float32), dtype=np.float32, block=g)
    if s2 is not None:
        u = (u * s2.astype(np.float32)).astype(np.float32)
    kappa = np.sqrt(np.float32(d // g), dtype=np.float32)  # correctly rounded; 1 when g = d
    with np.errstate(divide="ignore", invalid="ignore"):
        z = ((u * kappa).astype(np.float32) / n[..., None]).astype(np.float32)
    k = np.zeros(z.shape, dtype=np.int64)
    for t in thresholds:
        k += (z >= t).astype(np.int64)
    zero = (n == 0)[..., None]
    k = np.where(zero, levels // 2 - 1, k)  # stores sign 0, magnitude 0
    return k, n.astype(np.float16)


def _sign_magnitude(k, levels):
    """Split a level index k into (sign, magnitude): sign = k >= L/2, magnitude counts
    outward from the middle of the codebook on each side."""
    half = levels // 2
    sign = k >= half
    mag = np.where(sign, k - half, half - 1 - k)
    return sign.astype(np.uint8), mag.astype(np.uint8)


def encode_tier(x: np.ndarray, sign_words, bits: int):
    """Quantise fp16 rows ``x[..., D]`` with the ``bits``-bit tier (2, 3 or 4).

    Returns ``(planes tuple of uint8 arrays, norms float16 [...])``; the planes are
    TQ2: (2-bit sign-magnitude fields,); TQ3: (magnitude 2-bit, sign 1-bit);
    TQ4: (4-bit sign-magnitude fields,).
    """
    levels = 1 << bits
    k, norms = level_index(x, sign_words, levels)
    sign, mag = _sign_magnitude(k, levels)
    if bits == 2:
        return (pack_bits((sign << 1) | mag, 2),), norms
    if bits == 3:
        return (pack_bits(mag, 2), pack_bits(sign, 1)), norms
    if bits == 4:
        return (pack_bits((sign << 3) | mag, 4),), norms
    raise ValueError("bits must be 2, 3 or 4")


def codes_from_tier_planes(planes, d: int, bits: int) -> np.ndarray:
    """Level index k in 0..2^bits - 1 from a tier's planes."""
    half = 1 << (bits - 1)
    if bits == 2:
        f = unpack_bits(planes[0], 2, d).astype(np.int64)
        sign, mag = f >> 1, f & 1
    elif bits == 3:
        mag = unpack_bits(planes[0], 2, d).astype(np.int64)
        sign = unpack_bits(planes[1], 1, d).astype(np.int64)
    elif bits == 4:
        f = unpack_bits(planes[0], 4, d).astype(np.int64)
        sign, mag = f >> 3, f & 7
    else:
        raise ValueError("bits must be 2, 3 or 4")
    return np.where(sign == 1, half + mag, half - 1 - mag)


def decode_tier(planes, norms, sign_words, d: int, bits: int) -> np.ndarray:
    """Dequantise a tier to float64: x_hat = n16 * s1 .* blockdiag(H_G)(s2 .* c[k]) /
    sqrt(D G), which is (n16 / D) * s .* (H c[k]) for the first form."""
    levels, _ = codebook(1 << bits)
    ck = levels.astype(np.float64)[codes_from_tier_planes(planes, d, bits)]
    s1, s2, g = _rotation(sign_words, d)
    if s2 is not None:
        ck = ck * s2
    n = np.asarray(norms).astype(np.float64)[..., None]
    return (n / np.sqrt(float(d) * g)) * s1 * fwht(ck, dtype=np.float64, block=g)


def encode(x: np.ndarray, sign_words):
    """Quantise fp16 rows ``x[..., D]`` with TQ3.

    Returns ``(lo2 uint8 [..., D/4], hi1 uint8 [..., D/8], norms float16 [...])``.
    """
    (lo2, hi1), norms = encode_tier(x, sign_words, 3)
    return lo2, hi1, norms


def pack_bits(vals: np.ndarray, width: int) -> np.ndarray:
    """Pack small unsigned fields little-endian: element i at bit width * i of the row."""
    per = 8 // width
    d = vals.shape[-1]
    v = vals.reshape(vals.shape[:-1] + (d // per, per)).astype(np.uint32)
    out = np.zeros(v.shape[:-1], dtype=np.uint32)
    for j in range(per):
        out |= v[..., j] << (width * j)
    return out.astype(np.uint8)


def unpack_bits(packed: np.ndarray, width: int, d: int) -> np.ndarray:
    """Inverse of ``pack_bits``: the ``d`` fields of ``width`` bits of each row."""
    per = 8 // width
    p = np.asarray(packed).astype(np.uint32)
    mask = (1 << width) - 1
    parts = [(p >> (width * j)) & mask for j in range(per)]
    v = np.stack(parts, axis=-1)
    return v.reshape(p.shape[:-1] + (d,)).astype(np.uint8)


def codes_from_planes(lo2: np.ndarray, hi1: np.ndarray, d: int) -> np.ndarray:
    """TQ3 level index k in 0..7 from the two planes."""
    return codes_from_tier_planes((lo2, hi1), d, 3)


def decode(lo2, hi1, norms, sign_words, d: int) -> np.ndarray:
    """Dequantise TQ3 to float64 (see ``decode_tier``)."""
    return decode_tier((lo2, hi1), norms, sign_words, d, 3)


def bytes_per_value(d: int, bits: int = 3) -> float:
    """Storage per value: the tier's planes + one fp16 norm per vector."""
    plane_bytes = {2: d // 4, 3: d // 4 + d // 8, 4: d // 2}[bits]
    return (plane_bytes + 2) / d
