"""Pins of the oracle's E4M3 decoder against the OCP FP8 definition.

Known codes from the format's definition (bias 7, 3 fraction bits, no
infinities, S.1111.111 = NaN, max 448), monotonicity over the positive codes,
sign symmetry, and a round trip through the generator's independent encoder.
"""
import math

import numpy as np

import synth
from oracle import fp8


def test_known_codes():
    assert fp8.decode(0x00) == 0.0 and math.copysign(1, fp8.decode(0x80)) == -1
    assert fp8.decode(0x01) == 2.0 ** -9            # smallest subnormal
    assert fp8.decode(0x07) == 7 * 2.0 ** -9        # largest subnormal
    assert fp8.decode(0x08) == 2.0 ** -6            # smallest normal
    assert fp8.decode(0x38) == 1.0
    assert fp8.decode(0x39) == 1.125
    assert fp8.decode(0x40) == 2.0
    assert fp8.decode(0x7E) == 448.0 and fp8.decode(0xFE) == -448.0
    assert math.isnan(fp8.decode(0x7F)) and math.isnan(fp8.decode(0xFF))
    assert fp8.decode(0x78) == 256.0                # exponent field 15 is finite


def test_monotone_and_symmetric():
    pos = fp8.TABLE[:0x7F]
    assert np.all(np.diff(pos) > 0)
    np.testing.assert_array_equal(fp8.TABLE[0x80:0xFF], -pos)
    assert len(set(pos.tolist())) == 127


def test_round_trip_through_generator_encoder():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = fp8.decode(c)
        assert synth.e4m3_encode(v) == c, hex(c)
