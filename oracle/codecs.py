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

def e4m3_decode(codes) -> np.ndarray:
    """e4m3 bytes (any integer array) -> fp64 values."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.int64) & 0xFF]


def e4m3_encode(x) -> np.ndarray:
    """Values (fp32 or fp64) -> e4m3 bytes, RNE with saturation to +-448.

    Straight from the field layout: a magnitude below 2^-6 is subnormal and its
    code is its multiple of 2^-9 rounded half-to-even; otherwise, writing
    ``|x| = 2^e * (1 + f)`` with ``f`` in [0, 1), the 3-bit mantissa is ``8 f``
    rounded half-to-even (a carry to 8 bumps the exponent) and the code is
    ``(e + 7) << 3 | mantissa``. Magnitudes of 448 and above saturate to 448
    (code 0x7E). The sign bit is copied, so -0 and tiny negatives encode as
    0x80; NaN encodes as 0x7F. ``np.rint`` rounds half to even, and every
    scaling here is by a power of two, so no step rounds twice.
    """
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    finite_mag = np.where(np.isnan(mag) | (mag >= E4M3_MAX), 0.0, mag)
    sub = finite_mag < 2.0 ** -6
    code_sub = np.rint(finite_mag * 2.0 ** 9)                 # 0..8; 8 is the smallest normal
    frac, exp2 = np.frexp(finite_mag)                          # finite_mag = frac * 2^exp2, frac in [0.5, 1)
    e = exp2 - 1
    man = np.rint((2.0 * frac - 1.0) * 8.0)
    carry = man == 8.0
    e = np.where(carry, e + 1, e)
    man = np.where(carry, 0.0, man)
    code_norm = ((e + 7) << 3) + man.astype(np.int64)
    code = np.where(sub, code_sub.astype(np.int64), code_norm)
    code = np.where(mag >= E4M3_MAX, 126, np.minimum(code, 126))
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


# ----------------------------------------------------------------------------
# OCP Microscaling (MX) formats: FP4 E2M1 elements and E8M0 shared scales
# ----------------------------------------------------------------------------
#
# The V4.1 review names an MXFP4 indexer cache ("功能与动机"; the
# indexer_kv_dtype "mxfp4" switch of "风险与影响") without printing the format;
# MXFP4 is the OCP Microscaling format with FP4 E2M1 elements. For a 4-bit code
# ``s ee m``: ``ee == 0`` is subnormal, value ``(-1)^s * 0.5 * m``; otherwise
# ``(-1)^s * 2^(ee - 1) * (1 + m/2)``. The eight magnitudes are 0, 0.5, 1, 1.5, 2,
# 3, 4, 6; there is no infinity or NaN. E8M0 is an unsigned exponent: code c is
# ``2^(c - 127)``, code 255 is NaN.

E2M1_MAX = 6.0


def _e2m1_value(code: int) -> float:
    sign = (code >> 3) & 1
    exp = (code >> 1) & 0x3
    man = code & 0x1
    mag = 0.5 * man if exp == 0 else 2.0 ** (exp - 1) * (1.0 + man / 2.0)
    return -mag if sign else mag


#: value of every 4-bit code 0..15 as fp64
E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def e2m1_decode(codes) -> np.ndarray:
    """4-bit e2m1 codes (any integer array; the low nibble is used) -> fp64 values."""
    return E2M1_TABLE[np.asarray(codes, dtype=np.int64) & 0xF]


def e2m1_encode(x) -> np.ndarray:
    """Values -> e2m1 codes, round to nearest with ties to the even code, saturating to +-6.

    From the field layout: magnitudes below 1 are subnormal, multiples of 0.5
    rounded half-to-even (0.25 -> 0, 0.75 -> 1.0 whose mantissa bit is even);
    otherwise ``|x| = 2^e (1 + f)`` with the 1-bit mantissa ``2 f`` rounded
    half-to-even (a carry bumps the exponent). Magnitudes of 6 and above
    saturate to 6 (code 0b0111). The sign bit is copied. NaN is not accepted.
    """
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("e2m1 has no NaN")
    mag = np.minimum(np.abs(x), E2M1_MAX)
    sub = mag < 1.0
    m_sub = np.rint(mag * 2.0)                   # 0, 1 or 2 (2 = the smallest normal, 1.0)
    code_sub = np.where(m_sub == 2.0, 0b010, m_sub.astype(np.int64))
    frac, exp2 = np.frexp(np.where(sub, 1.0, mag))   # mag = frac * 2^exp2, frac in [0.5, 1)
    e = exp2 - 1                                  # 0, 1 or 2
    man = np.rint((2.0 * frac - 1.0) * 2.0)       # 0, 1 or 2 (carry)
    carry = man == 2.0
    e = np.where(carry, e + 1, e)
    man = np.where(carry, 0.0, man)
    code_norm = ((e + 1) << 1) + man.astype(np.int64)
    code = np.where(sub, code_sub, np.minimum(code_norm, 0b0111))
    return (code | (np.signbit(x).astype(np.int64) << 3)).astype(np.uint8)


def e8m0_decode(codes) -> np.ndarray:
    """E8M0 scale codes -> fp64 values ``2^(c - 127)``; 255 -> NaN."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    return np.where(c == 255, np.nan, np.ldexp(1.0, c - 127))
