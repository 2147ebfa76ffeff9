"""Code decoders for the oracle (test infrastructure; see package docstring).

* FP8 E4M3 (OCP 8-bit floating point, "E4M3" variant used by MXFP8 and by the
  pages' FP8 activations and weights): 1 sign bit, 4 exponent bits with bias 7,
  3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is
  NaN; there are no infinities; the largest finite magnitude is 448.
* UE8M0 (the MX block-scale format): 8 unsigned exponent bits, value
  2^(e-127); 0xFF is NaN.
* FP8 E5M2 (OCP 8-bit floating point, "E5M2"): 1 sign bit, 5 exponent bits with
  bias 15, 2 mantissa bits; exponent field 0 is subnormal (m/4 * 2^-14); exponent
  field 31 is infinity (m = 0) or NaN; the largest finite magnitude is 57344.
* bfloat16: the top 16 bits of an IEEE binary32.
* float16: IEEE binary16.

All decoders return float64 arrays; the decode is exact.  ``encode_fp8`` rounds
a real value to the nearest finite E4M3 / E5M2 value, ties to the even code,
saturating at the largest finite magnitude (the "satfinite" conversion).
"""
from __future__ import annotations

import numpy as np


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    normal = (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0)
    subnormal = (man / 8.0) * 2.0 ** -6
    mag = np.where(exp == 0, subnormal, normal)
    mag = np.where((exp == 0xF) & ((c & 0x7) == 0x7), np.nan, mag)
    return sign * mag


def decode_ue8m0(codes: np.ndarray) -> np.ndarray:
    e = np.asarray(codes, dtype=np.uint8).astype(np.float64)
    return np.where(e == 255, np.nan, np.exp2(e - 127.0))


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):  # NaN sentinels decode to NaN silently
        return b.view(np.float32).astype(np.float64)


def decode_e5m2(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 2) & 0x1F
    man = (c & 0x3).astype(np.float64)
    normal = (1.0 + man / 4.0) * np.exp2(exp.astype(np.float64) - 15.0)
    subnormal = (man / 4.0) * 2.0 ** -14
    mag = np.where(exp == 0, subnormal, normal)
    mag = np.where(exp == 31, np.where((c & 0x3) == 0, np.inf, np.nan), mag)
    return sign * mag


def decode_fp16(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


# finite non-negative magnitudes of each FP8 format, in code order (they increase with the code)
_FP8_MAGS = {"e4m3": decode_e4m3(np.arange(0x7F, dtype=np.uint8)),   # 0x00..0x7E, max 448
             "e5m2": decode_e5m2(np.arange(0x7C, dtype=np.uint8))}   # 0x00..0x7B, max 57344


def encode_fp8(v: np.ndarray, fmt: str) -> np.ndarray:
    """Real values -> FP8 codes of ``fmt`` ("e4m3" or "e5m2"): nearest finite value,
    ties to the even code (mantissa LSB 0), magnitudes beyond the largest finite
    value saturate to it, the sign bit taken from the input."""
    mags = _FP8_MAGS[fmt]
    top = len(mags) - 1
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), mags[-1])
    hi = np.clip(np.searchsorted(mags, a, side="left"), 0, top)
    lo = np.clip(hi - 1, 0, top)
    d_lo, d_hi = a - mags[lo], mags[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return (code | (np.signbit(v).astype(np.uint8) << np.uint8(7))).astype(np.uint8)


def fp8_neighbours(v: np.ndarray, fmt: str):
    """The FP8 codes just below and just above |v| (with v's sign) and the midpoint
    between them, for comparing a code rounded from a slightly different value."""
    mags = _FP8_MAGS[fmt]
    top = len(mags) - 1
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), mags[-1])
    hi = np.clip(np.searchsorted(mags, a, side="left"), 0, top)
    lo = np.clip(hi - 1, 0, top)
    sign = np.signbit(v).astype(np.uint8) << np.uint8(7)
    return ((lo.astype(np.uint8) | sign), (hi.astype(np.uint8) | sign), (mags[lo] + mags[hi]) / 2)
