"""Row FP8 quantisation of the activation (test infrastructure; see package docstring).

AWS Neuron "Kernel reference: qkv_cte", section "Interface": the projection's
input is a row-packed activation [B, S, H + 4] -- H FP8 (E4M3) codes followed by
a 4-byte fp32 dequantisation scale per row -- made from the bf16 hidden state by
a row quantiser (row_quantize_packed); the projection kernel itself does not
quantise.  The page names the operation and its output layout but gives no
formula.  The reading used here is symmetric absmax scaling onto the E4M3 range,
with the code defined by the layout's own dequantisation identity: the row
stores one fp32 scale, and x is recovered as code * scale, so the code is x
divided by that stored scale, rounded to E4M3:

    m[t]      = max(max_h |x[t, h]|, 2^-100)      (exact: x is bf16; the floor keeps
                                                  the scale a normal fp32 number for rows
                                                  of zeros or of bf16 subnormals)
    scale[t]  = m[t] / 448                        fp32, rounded to nearest -- the stored scale
    code[t,h] = E4M3(x[t, h] / scale[t])          the fp32 quotient (IEEE division, rounded to
                                                  nearest), then rounded to E4M3 half-to-even,
                                                  saturated to +-448, the sign of zero kept

The codes are integers that floating point decides, so every step is taken in
fp32, the type of the stored scale (numpy float32 arithmetic is IEEE binary32
with round-to-nearest-even, division included).
"""
from __future__ import annotations

import numpy as np

from .codes import decode_bf16, decode_e4m3

E4M3_MAX = 448.0
AMAX_FLOOR = 2.0 ** -100

# the 127 non-negative finite E4M3 magnitudes, in code order (codes 0x00..0x7E);
# they increase with the code
_E4M3_MAGS = decode_e4m3(np.arange(127, dtype=np.uint8))


def encode_e4m3_rne_sat(v: np.ndarray) -> np.ndarray:
    """float32 -> E4M3 code: nearest representable magnitude, ties to the even code
    (mantissa LSB 0), magnitudes above 448 saturate to 448, sign bit from the input."""
    v = np.asarray(v, dtype=np.float32)
    a = np.minimum(np.abs(v).astype(np.float64), E4M3_MAX)
    hi = np.clip(np.searchsorted(_E4M3_MAGS, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_lo = a - _E4M3_MAGS[lo]
    d_hi = _E4M3_MAGS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag_code = np.where(pick_hi, hi, lo).astype(np.uint8)
    sign = np.signbit(v).astype(np.uint8) << np.uint8(7)
    return (mag_code | sign).astype(np.uint8)


def row_quantize(x_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """bf16 bit patterns [T, H] -> (E4M3 codes [T, H] uint8, dequant scale [T] float32)."""
    x = decode_bf16(np.asarray(x_bits, dtype=np.uint16)).astype(np.float32)
    m = np.maximum(np.max(np.abs(x), axis=1), np.float32(AMAX_FLOOR)).astype(np.float32)
    scale = (m / np.float32(E4M3_MAX)).astype(np.float32)
    quot = (x / scale[:, None]).astype(np.float32)
    return encode_e4m3_rne_sat(quot), scale


def row_quantize_packed(x_bits: np.ndarray) -> np.ndarray:
    """The page's row-packed layout [T, H + 4]: the codes, then the scale's 4 bytes
    (little-endian IEEE binary32)."""
    codes, scale = row_quantize(x_bits)
    tail = scale.astype("<f4").view(np.uint8).reshape(-1, 4)
    return np.concatenate([codes, tail], axis=1)
