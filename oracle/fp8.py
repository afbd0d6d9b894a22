"""Oracle FP8 E4M3 quantisation of K/V for a pool that stores 8-bit floats.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages keep K/V in fp16; an 8-bit pool is one of the variants their
tuning discussion leaves open (other model configurations, [CA-summary §7]).
The format is the published E4M3 encoding of the OCP 8-bit floating point
specification, restated here from its definition:

    code = s eeee mmm  (sign, 4 exponent bits with bias 7, 3 mantissa bits)
    e > 0:  value = (-1)^s * 2^(e - 7) * (1 + m / 8)
    e = 0:  value = (-1)^s * 2^(-6) * (m / 8)          (subnormals, and +-0)
    e = 15 and m = 7 is NaN; there are no infinities; the largest finite
    magnitude is 2^8 * 1.75 = 448.

Quantising a stored element x (fp16) with the pool's scale (reading R14):
    y = fp32(x) * fp32(1 / scale)           (both roundings IEEE fp32)
    code = the finite E4M3 value nearest to y, ties to the even code
           (mantissa bit 0 clear); |y| beyond 448 gives +-448 (saturation)
and the element attention sees is decode(code) * scale, exactly, in fp64.

Pins (tests/test_oracle_fp8.py): the definition's landmark values, rounding
ties, subnormals and saturation by hand; every encode against brute force
over all 254 finite codes; in-range values against torch's float8_e4m3fn
cast (a library routine).
"""
from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0


def _code_values() -> np.ndarray:
    """Value of each of the 256 codes (NaN for the two NaN codes)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 15 and m == 7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = s * 2.0 ** -6 * (m / 8.0)
        else:
            vals[code] = s * 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return vals


CODE_VALUES = _code_values()
# non-negative finite codes in increasing value (0x00 .. 0x7E)
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = CODE_VALUES[:0x7F]


def decode(codes) -> np.ndarray:
    """float64 value of each code."""
    return CODE_VALUES[np.asarray(codes, dtype=np.uint8).astype(np.int64)]


def encode(y) -> np.ndarray:
    """Nearest E4M3 code to each float32 ``y`` (ties to the even code),
    saturating beyond +-448.  NaN input is not expected and is rejected."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    if np.isnan(y).any():
        raise ValueError("NaN input")
    a = np.minimum(np.abs(y), MAX_FINITE)
    hi = np.searchsorted(_POS_VALUES, a, side="left")          # first value >= a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    mag = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo])
    # the sign is kept, also when the magnitude rounds to zero (-0 is 0x80)
    return (mag | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def inverse_scale(scale: float) -> np.float32:
    """fp32(1 / scale), as the quantiser multiplies by it."""
    return np.float32(1.0) / np.float32(scale)


def quantize(x, scale: float) -> np.ndarray:
    """Codes of fp16 elements ``x`` under ``scale`` (reading R14)."""
    x32 = np.asarray(x, dtype=np.float16).astype(np.float32)
    return encode(x32 * inverse_scale(scale))


def dequantize(codes, scale: float) -> np.ndarray:
    """The elements attention sees: code value times scale, float64."""
    return decode(codes) * float(np.float32(scale))
