"""FP8 latent rows: E4M3 codes with one fp32 scale a row -- TEST INFRASTRUCTURE ONLY.

Issue #1313, step 1.3, item 3: FP8 latent rows on pages, a page's fp32 row scales stored
behind its 512 rows (516 latent bytes a row and cache).  The pages fix neither the
FP8 format nor how the scale is chosen.  Read here as the OCP E4M3 format (1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits; subnormals; no infinities; 0x7F / 0xFF are NaN;
the largest finite value is 448) and a per-row absolute-maximum scale:
  scale = amax / 448 (fp32 division), code_i = E4M3(x_i / scale) (fp32 division, then
  round to nearest, ties to even, saturating to +-448); a row of zeros stores scale 0, codes 0.
The latent value a code stands for is decode(code) * scale, exactly (in float64).

Where floating point decides a code, this module takes the decision in fp32, as the
quantizer does.  Encoding and decoding follow the bit fields of the format, not a library;
encode() is the scalar definition and encode_array() the same rule over arrays (pinned to it).
"""
from __future__ import annotations

import math

import numpy as np

MAX_FINITE = 448.0
NAN_CODE = 0x7F


def decode(code: int) -> float:
    """The value of one E4M3 code."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 0xF and m == 7:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** -9           # subnormal: m/8 * 2^(1-7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _round_half_even(v: float) -> int:
    f = math.floor(v)
    d = v - f
    if d > 0.5 or (d == 0.5 and f % 2 == 1):
        return int(f) + 1
    return int(f)


def encode(x: float) -> int:
    """E4M3 code of x: round to nearest, ties to even, saturating to +-448; NaN -> 0x7F."""
    x = float(np.float32(x))
    if math.isnan(x):
        return NAN_CODE
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if a >= MAX_FINITE:
        return sign | 0x7E
    if a < 2.0 ** -6:                          # subnormal range: steps of 2^-9
        m = _round_half_even(a / 2.0 ** -9)    # exact: a is an fp32 value, the ratio a power of 2
        return sign | m if m < 8 else sign | 0x08
    e = math.floor(math.log2(a))
    while 2.0 ** e > a:                        # guard log2 rounding
        e -= 1
    while 2.0 ** (e + 1) <= a:
        e += 1
    m = _round_half_even((a / 2.0 ** e - 1.0) * 8.0)
    if m == 8:
        e, m = e + 1, 0
    if e > 8 or (e == 8 and m == 7):           # past 448 after rounding
        return sign | 0x7E
    return sign | ((e + 7) << 3) | m


def encode_array(x) -> np.ndarray:
    """encode() of every value of an array, the same definition written with numpy: the
    exponent from frexp, the 3-bit mantissa rounded half to even (rint), the subnormal range
    in steps of 2^-9, saturation to +-448 and NaN -> 0x7F.  uint8 codes."""
    v = np.asarray(x, dtype=np.float32).astype(np.float64)
    nan = np.isnan(v)
    a = np.minimum(np.where(nan, 0.0, np.abs(v)), 2.0 * MAX_FINITE)   # all past 448 saturate
    sign = np.where(np.signbit(v), 0x80, 0).astype(np.int64)
    ms = np.rint(a / 2.0 ** -9).astype(np.int64)                 # subnormal: exact ratio
    sub_code = np.where(ms >= 8, 0x08, ms)
    fm, fe = np.frexp(a)                                         # a = fm * 2^fe, fm in [0.5, 1)
    e = fe.astype(np.int64) - 1
    mm = np.rint((2.0 * fm - 1.0) * 8.0).astype(np.int64)        # exact before rounding
    carry = mm == 8
    e = np.where(carry, e + 1, e)
    mm = np.where(carry, 0, mm)
    norm_code = ((e + 7) << 3) | mm
    over = (a >= MAX_FINITE) | (e > 8) | ((e == 8) & (mm == 7))
    code = np.where(a < 2.0 ** -6, sub_code, np.where(over, 0x7E, norm_code))
    code = np.where(nan, NAN_CODE, code | sign)
    return code.astype(np.uint8)


def quantize_row(x) -> tuple:
    """(codes uint8[n], scale float32) of one latent row x (float32 values, finite)."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    if amax == 0:
        return np.zeros(x.size, np.uint8), np.float32(0)
    scale = np.float32(amax / np.float32(MAX_FINITE))
    q = (x / scale).astype(np.float32)
    return encode_array(q), scale


def dequantize_row(codes, scale) -> np.ndarray:
    """float64 values decode(code) * scale, exactly."""
    return np.array([decode(c) for c in np.asarray(codes, np.uint8)], np.float64) * float(np.float32(scale))


_TABLE = None


def decode_table() -> np.ndarray:
    """float64 value of every code (NaN for 0x7F and 0xFF)."""
    global _TABLE
    if _TABLE is None:
        _TABLE = np.array([decode(c) for c in range(256)], np.float64)
    return _TABLE


def quantize_rows(x) -> tuple:
    """quantize_row over the last axis of a [..., n] array: (codes uint8[..., n], scales float32[...])."""
    x = np.asarray(x, dtype=np.float32)
    flat = x.reshape(-1, x.shape[-1])
    amax = np.max(np.abs(flat), axis=1).astype(np.float32) if flat.size else np.zeros(flat.shape[0], np.float32)
    scales = (amax / np.float32(MAX_FINITE)).astype(np.float32)
    safe = np.where(scales == 0, np.float32(1), scales).astype(np.float32)
    q = (flat / safe[:, None]).astype(np.float32)
    codes = np.where((scales == 0)[:, None], np.uint8(0), encode_array(q))
    return codes.reshape(x.shape), scales.reshape(x.shape[:-1])


def dequantize_rows(codes, scales) -> np.ndarray:
    """float64 [..., n] values of quantize_rows' output."""
    t = decode_table()[np.asarray(codes, np.uint8)]
    return t * np.asarray(scales, np.float32).astype(np.float64)[..., None]
