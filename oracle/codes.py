"""Code decoders for the oracle (test infrastructure; see package docstring).

* FP8 E4M3 (OCP 8-bit floating point, "E4M3" variant used by MXFP8 and by the
  pages' FP8 activations and weights): 1 sign bit, 4 exponent bits with bias 7,
  3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is
  NaN; there are no infinities; the largest finite magnitude is 448.
* UE8M0 (the MX block-scale format): 8 unsigned exponent bits, value
  2^(e-127); 0xFF is NaN.
* bfloat16: the top 16 bits of an IEEE binary32.

All decoders return float64 arrays; the decode is exact.
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
