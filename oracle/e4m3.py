"""FP8 E4M3 codec written from the OCP 8-bit floating point definition.

E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
  exponent field 0      -> subnormal, value = m * 2**-9
  exponent field 1..15  -> normal, value = (1 + m/8) * 2**(e - 7)
  code 0x7F / 0xFF      -> NaN (there is no infinity); largest finite 0x7E = 448.

Encoding used by the method's activation quantisation: round to nearest,
ties to even (the even code has mantissa LSB 0), saturating to +-448 instead of
producing NaN.  Saturation before the e4m3 cast is what the SGLang PR #37796
page ("moe_wna16: 2-bit experts ...", Modifications, mem_cache/memory_pool.py
fp8 write path) does, because an unsaturated cast returns NaN beyond the range.
The sign is kept, so a negative value that rounds to zero encodes as 0x80.
"""
from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0


def _decode_one(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


# value of every code, float64
DECODE_TABLE = np.array([_decode_one(c) for c in range(256)], dtype=np.float64)
# the 127 non-negative finite values, codes 0x00 .. 0x7E, in increasing order
_POS_VALUES = DECODE_TABLE[:0x7F].copy()


def decode(codes) -> np.ndarray:
    """E4M3 codes (uint8) -> float64 values."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def encode(x) -> np.ndarray:
    """float -> E4M3 code, round to nearest even, saturating at +-448, sign kept.

    The rounding is decided on the exact value of ``x`` (float32 or float64
    inputs are both exact in float64).
    """
    x = np.asarray(x)
    xd = x.astype(np.float64)
    mag = np.abs(xd)
    nan = np.isnan(mag)
    mag = np.where(nan, 0.0, np.minimum(mag, MAX_FINITE))
    hi = np.searchsorted(_POS_VALUES, mag, side="left")  # first value >= mag
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS_VALUES[hi] - mag
    d_lo = mag - _POS_VALUES[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(mag == _POS_VALUES[hi], hi, code).astype(np.uint8)
    code = code | np.where(np.signbit(xd), np.uint8(0x80), np.uint8(0))
    code = np.where(nan, np.uint8(0x7F), code)
    return code.astype(np.uint8)
