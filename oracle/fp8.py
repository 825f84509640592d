"""OCP 8-bit floating point E4M3 decoding (oracle).

The fp8 expert format is named only as "fp8_block" on the page "FreeToken: az
VRAM ile büyük MoE modelleri" (section "Tuzaklar", the bandwidth printout).
Reading: OCP FP8 E4M3 codes (OCP 8-bit Floating Point Specification, v1.0):
1 sign bit, 4 exponent bits with bias 7, 3 fraction bits; exponent field 0 is
subnormal (fraction/8 * 2^-6); the code S.1111.111 is NaN; there are no
infinities; the largest finite magnitude is 1.75 * 2^8 = 448.
"""
from __future__ import annotations

import math

import numpy as np


def decode(code: int) -> float:
    code &= 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    frac = code & 0x7
    if exp == 0xF and frac == 0x7:
        return math.nan
    if exp == 0:
        return sign * (frac / 8.0) * 2.0 ** -6
    return sign * (1.0 + frac / 8.0) * 2.0 ** (exp - 7)


TABLE = np.array([decode(c) for c in range(256)], dtype=np.float64)


def decode_array(codes: np.ndarray) -> np.ndarray:
    return TABLE[np.asarray(codes, dtype=np.uint8)]
