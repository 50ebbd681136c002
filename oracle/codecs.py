"""Narrow number formats used by the indexer, decoded and encoded from their definitions.

Test infrastructure (see the package docstring): only tests, smoke and the
benchmark's CPU-baseline leg use it.

FP8 e4m3 (OCP 8-bit floating point, E4M3 variant). The pages only say "FP8"
(DSA explainer, cost table: the indexer stores FP8; step ④ quantises q to FP8
with one scale per 128 elements); the e4m3 flavour is the one the indexer cache
uses. Definition, for a byte ``b = s eeee mmm``:

* ``e == 0``: subnormal, value ``(-1)^s * 2^-6 * m/8``
* ``0 < e``: normal, value ``(-1)^s * 2^(e-7) * (1 + m/8)``
* ``e == 15 and m == 7``: NaN (0x7F / 0xFF); there are no infinities,
  so the largest finite magnitude is ``2^8 * 1.75 = 448``.

Encoding is round-to-nearest, ties-to-even, saturating to +-448 (every finite
input maps to a finite code). NaN encodes as 0x7F.

bf16 is the upper 16 bits of an IEEE binary32 value. Decoding shifts them back;
encoding rounds the lower 16 bits away, to nearest with ties to even. The V4.1
review states this for the bf16 per-head weights: the bf16 value equals the
fp32 result rounded once (实现拆解 item 5 and the test list).
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _e4m3_value(code: int) -> float:
    """Value of one e4m3 byte, straight from the format definition."""
    sign = (code >> 7) & 1
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        mag = (man / 8.0) * 2.0 ** -6
    else:
        mag = (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return -mag if sign else mag


#: value of every byte 0..255 as fp64 (NaN for 0x7F and 0xFF)
E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)

# Codes 0x00..0x7E are the non-negative finite values in strictly increasing order
# (the byte order of a sign-magnitude float with a monotone exponent field).
_E4M3_POS = E4M3_TABLE[:127].copy()


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 bytes (any integer array) -> fp64 values."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.int64) & 0xFF]


def e4m3_encode(x) -> np.ndarray:
    """Values (fp32 or fp64) -> e4m3 bytes, RNE with saturation to +-448.

    The nearest representable magnitude is found by bracketing ``|x|`` between
    two consecutive codes; an exact midpoint goes to the even code (its mantissa
    LSB is the byte's LSB). The sign bit is copied, so -0 and tiny negatives
    encode as 0x80.
    """
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    finite_mag = np.where(np.isnan(mag), 0.0, mag)
    lo = np.searchsorted(_E4M3_POS, finite_mag, side="right") - 1
    lo = np.clip(lo, 0, 126)
    hi = np.minimum(lo + 1, 126)
    d_lo = finite_mag - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - finite_mag
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((lo & 1) == 1))
    code = np.where(take_hi, hi, lo)
    code = np.where(finite_mag >= E4M3_MAX, 126, code)
    code = code | (np.signbit(x).astype(np.int64) << 7)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def bf16_decode(u16) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    u = np.asarray(u16, dtype=np.uint32) & 0xFFFF
    return (u << 16).astype(np.uint32).view(np.float32)


def bf16_encode(x) -> np.ndarray:
    """fp32 values -> bf16 bit patterns, round to nearest, ties to even. NaN -> quiet NaN."""
    f = np.array(x, dtype=np.float32)
    u = f.reshape(-1).view(np.uint32).astype(np.uint64).reshape(f.shape)
    upper = u >> 16
    lower = u & 0xFFFF
    round_up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & 1) == 1))
    out = upper + round_up.astype(np.uint64)
    nan_bits = (upper & 0x8000) | 0x7FC0
    out = np.where(np.isnan(f), nan_bits, out)
    return out.astype(np.uint16)
