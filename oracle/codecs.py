"""Storage-format codecs: bf16 / fp16 / fp8-e4m3 bit patterns <-> float64.

Test infrastructure (see ``oracle/__init__``).

[P2] §"KV量子化: FP8とINT8" states that the KV cache may be stored as FP8 at
one byte per element (about half of FP16).  The pages do not spell out the FP8
encoding; the format used is E4M3 as defined by the OCP 8-bit floating point
specification (OFP8): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
bits, subnormals when the exponent field is 0, no infinities, and the two
codes S.1111.111 reserved for NaN.  The largest finite magnitude is
1.75 * 2**8 = 448.

Quantisation ("satfinite", round-to-nearest-even) is written here from that
definition alone: the finite non-negative E4M3 values are enumerated, the
nearest one is chosen, ties go to the code whose mantissa LSB is 0, and any
magnitude at or above 448 (including +-inf) saturates to 448.

INT8 with a scale and a zero point (the same section lists INT8 KV at one
byte per element that "needs a scale / zero point", without a formula): the
plainest affine reading is value = (code - zero_point) * scale with a signed
8-bit code in [-128, 127] and an integer zero point, one (scale, zero_point)
pair per KV head for K and one for V.  Quantisation of a float32 product
y = x * inv_scale (formed in float32 by the caller): code = clamp(rne(y) +
zero_point, -128, 127), where rne rounds to the nearest integer with ties to
even; +-inf saturate, and NaN is taken to saturate to +127.

Pins: ``tests/test_oracle_pins.py::test_e4m3_*`` (known OCP values, all 256
codes against torch.float8_e4m3fn, round trips, tie midpoints, saturation),
``test_bf16_*`` (against torch.bfloat16) and ``test_int8_*`` (round trips of
all codes for several zero points, ties to even, saturation, torch's
quantize_per_tensor with scale 1).
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
_E4M3_NAN_CODE = 0x7F


def _e4m3_magnitude(code7: int) -> float:
    """Value of the 7-bit magnitude field (exponent<<3 | mantissa); NaN for 0x7F."""
    e = (code7 >> 3) & 0xF
    m = code7 & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        # subnormal: 0.m * 2**(1 - bias) = m/8 * 2**-6
        return (m / 8.0) * 2.0 ** (1 - 7)
    return (1.0 + m / 8.0) * 2.0 ** (e - 7)


# Table of all 256 code values (index = code), built from the definition.
_E4M3_TABLE = np.array(
    [(-1.0 if (c & 0x80) else 1.0) * _e4m3_magnitude(c & 0x7F) for c in range(256)],
    dtype=np.float64,
)
# Finite non-negative magnitudes in code order 0x00..0x7E; they increase with the code.
_E4M3_POS = _E4M3_TABLE[:0x7F].copy()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """uint8 E4M3 codes -> float64 values (exact)."""
    codes = np.asarray(codes, dtype=np.uint8)
    return _E4M3_TABLE[codes.astype(np.int64)]


def e4m3_encode_f32(x: np.ndarray) -> np.ndarray:
    """float32 values -> uint8 E4M3 codes, round-to-nearest-even, saturating.

    The input is taken as float32 (the product x * inv_scale is formed in
    IEEE float32 before this call).  NaN maps to 0x7F.  The sign of the input
    is kept, including for results that round to zero.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    # index of the first table value >= a
    hi = np.searchsorted(_E4M3_POS, a, side="left")
    hi = np.clip(hi, 0, len(_E4M3_POS) - 1)
    lo = np.clip(hi - 1, 0, len(_E4M3_POS) - 1)
    v_hi = _E4M3_POS[hi]
    v_lo = _E4M3_POS[lo]
    d_hi = v_hi - a
    d_lo = a - v_lo
    # nearest; exact tie -> even code (mantissa LSB 0 == even code number)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= _E4M3_POS[-1], len(_E4M3_POS) - 1, code)  # satfinite
    code = np.where(a <= 0.0, 0, code)
    code = code.astype(np.uint8) | np.where(sign, 0x80, 0).astype(np.uint8)
    code = np.where(nan, _E4M3_NAN_CODE, code).astype(np.uint8)
    return code


def int8_decode(codes: np.ndarray, zero_point) -> np.ndarray:
    """int8 codes -> float64 (code - zero_point), exact; zero_point broadcasts."""
    c = np.asarray(codes, dtype=np.int8).astype(np.float64)
    return c - np.asarray(zero_point, dtype=np.int64).astype(np.float64)


def int8_encode_f32(y: np.ndarray, zero_point) -> np.ndarray:
    """float32 values (already x * inv_scale) -> int8 codes: clamp(rne(y) + zp, -128, 127)."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    zp = np.asarray(zero_point, dtype=np.int64).astype(np.float64)
    nan = np.isnan(y)
    r = np.rint(np.where(nan, 0.0, y)) + zp        # numpy rint: nearest, ties to even
    r = np.clip(r, -128.0, 127.0)
    r = np.where(nan, 127.0, r)
    return r.astype(np.int8)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16/int16) -> float64 (exact).

    bfloat16 is the upper half of an IEEE binary32 word.
    """
    b = np.asarray(bits).view(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f16_to_f64(x: np.ndarray) -> np.ndarray:
    """IEEE binary16 -> float64 (exact)."""
    return np.asarray(x, dtype=np.float16).astype(np.float64)


def storage_to_f64(x: np.ndarray, fmt: str) -> np.ndarray:
    """Decode a storage array ('f16', 'bf16' bits, 'e4m3' codes, 'f32') to float64."""
    if fmt == "f16":
        return f16_to_f64(x)
    if fmt == "bf16":
        return bf16_bits_to_f64(x)
    if fmt == "e4m3":
        return e4m3_decode(x)
    if fmt == "i8":
        return np.asarray(x, dtype=np.int8).astype(np.float64)   # raw codes (no zero point)
    if fmt == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown storage format {fmt!r}")


def storage_to_f32(x: np.ndarray, fmt: str) -> np.ndarray:
    """Decode a 16-bit storage array to float32 (exact widening)."""
    return storage_to_f64(x, fmt).astype(np.float32)
