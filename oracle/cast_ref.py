"""Element conversions of the fused permute + cast -- TEST INFRASTRUCTURE ONLY.

The TVM "permute_layout" page admits only equal source and destination dtypes
("What it accepts": a dtype mismatch is a reject reason).  The fused permute +
cast widens that rule: every element is moved as the page's permute moves it and
converted on the way.  The conversions are the IEEE 754 ones, written out here
from their definitions:

* binary32 -> binary16 and binary32 -> bfloat16 round to nearest, ties to even:
  the result is the representable value nearest to x on the target's grid
  (spacing 2**(e - p + 1) at binary exponent e, p significand bits; the
  subnormal spacing below the smallest normal exponent), a tie going to the
  candidate whose last significand bit is 0; results beyond the largest finite
  value become infinities of the same sign.
* binary16 -> binary32 and bfloat16 -> binary32 are exact.
* NaNs (a reading; IEEE 754 leaves payloads to the implementation): narrowing
  keeps the sign and the upper payload bits and, if those are all zero, sets the
  lowest payload bit so the result stays a NaN; widening keeps sign and payload
  (moved to the upper payload bits).

bfloat16 is the upper half of binary32: 1 sign bit, 8 exponent bits, 7 stored
significand bits.
"""
from __future__ import annotations

import numpy as np

CASTS = {"f32_to_bf16": (4, 2), "f32_to_f16": (4, 2), "bf16_to_f32": (2, 4),
         "f16_to_f32": (2, 4)}


def _round_to_grid(x64, p, emin, max_finite):
    """Nearest value to x64 (float64 array, exact binary32 values) on the grid of a
    binary format with p significand bits and smallest normal exponent emin, ties
    to even (np.rint rounds halves to even); overflow to +-inf."""
    ax = np.abs(x64)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        e = np.floor(np.log2(np.where((ax > 0) & np.isfinite(ax), ax, 1.0)))
    # log2 of an exact power of two can land a hair low/high: correct e so that
    # 2**e <= ax < 2**(e + 1)
    e = np.where(np.exp2(e) > ax, e - 1, e)
    e = np.where(np.exp2(e + 1) <= ax, e + 1, e)
    e = np.maximum(e, emin)                       # subnormals share the emin spacing
    ulp = np.exp2(e - (p - 1))
    v = np.rint(x64 / ulp) * ulp                  # exact: ulp is a power of two
    v = np.where(np.abs(v) > max_finite, np.copysign(np.inf, x64), v)
    return np.where((ax == 0) | np.isinf(x64), x64, v)     # zeros and infinities stay


def f32_to_f16_bits(u32):
    u32 = np.asarray(u32, dtype=np.uint32)
    x = u32.view(np.float32).astype(np.float64)
    nan = np.isnan(x)
    v = _round_to_grid(np.where(nan, 0.0, x), 11, -14, 65504.0)
    with np.errstate(over="ignore"):
        out = v.astype(np.float16).view(np.uint16)    # v is exactly representable
    sign = ((u32 >> 16) & 0x8000).astype(np.uint16)
    pay = ((u32 & 0x007FFFFF) >> 13).astype(np.uint16)
    nan_bits = sign | np.uint16(0x7C00) | np.where(pay == 0, np.uint16(1), pay)
    return np.where(nan, nan_bits, out).astype(np.uint16)


BF16_MAX = float(np.uint32(0x7F7F0000).view(np.float32))   # (2 - 2**-7) * 2**127


def f32_to_bf16_bits(u32):
    u32 = np.asarray(u32, dtype=np.uint32)
    x = u32.view(np.float32).astype(np.float64)
    nan = np.isnan(x)
    v = _round_to_grid(np.where(nan, 0.0, x), 8, -126, BF16_MAX)
    out = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # exact
    sign = ((u32 >> 16) & 0x8000).astype(np.uint16)
    pay = ((u32 & 0x007FFFFF) >> 16).astype(np.uint16)
    nan_bits = sign | np.uint16(0x7F80) | np.where(pay == 0, np.uint16(1), pay)
    return np.where(nan, nan_bits, out).astype(np.uint16)


def f16_to_f32_bits(u16):
    u16 = np.asarray(u16, dtype=np.uint16)
    h = u16.view(np.float16)
    out = h.astype(np.float32).view(np.uint32)     # exact for every non-NaN value
    u = u16.astype(np.uint32)
    nan_bits = ((u & 0x8000) << 16) | np.uint32(0x7F800000) | ((u & 0x03FF) << 13)
    return np.where(np.isnan(h), nan_bits, out).astype(np.uint32)


def bf16_to_f32_bits(u16):
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).astype(np.uint32)


CONVERT = {"f32_to_bf16": (np.uint32, f32_to_bf16_bits), "f32_to_f16": (np.uint32, f32_to_f16_bits),
           "bf16_to_f32": (np.uint16, bf16_to_f32_bits), "f16_to_f32": (np.uint16, f16_to_f32_bits)}


def convert_bytes(raw, cast):
    """Convert a byte buffer of source elements to a byte buffer of target elements."""
    src_t, fn = CONVERT[cast]
    return np.ascontiguousarray(fn(np.frombuffer(raw.tobytes(), dtype=src_t))).view(np.uint8)
