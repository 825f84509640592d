"""The fp8 block scales the parity cases feed the prefill GEMMs (CPU).

The prefill converter dequantises a tile's e4m3 weights with one fp16
multiply per pair when every block scale of the tile is an fp16 value, and
forms the product in fp32 otherwise (both round the exact product once).
These tests pin which route each GPU parity case takes: the generated banks
have only fp16-valued scales, and the shifted bank of
`test_fp8_prefill_parity_scales_off_fp16` has a scale off the fp16 grid in
every Wg and Wd row block, so every gate/up and down tile takes the fp32
route there.  They also check that the shift is the exact power-of-two
change of the weights it claims to be, through the oracle's decoding, and the
arithmetic the one-multiply route rests on: for every e4m3 value and bf16
scales on the fp16 grid, one rounding of the exact product to fp16.
"""
import numpy as np

import synth
from oracle import ffn as offn
from tests.harness import shift_fp8_scales
from tests.test_gpu_prefill import FP8_DSV4_DIMS_PREFILL, FP8_SMALL_PREFILL


def scales(blob: np.ndarray, H: int, I: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    g = (H // 128) * (I // 128)
    s = blob[3 * H * I:3 * H * I + 6 * g].view(np.uint16)
    v = (s.astype(np.uint32) << 16).view(np.float32)
    return (v[:g].reshape(I // 128, H // 128), v[g:2 * g].reshape(I // 128, H // 128),
            v[2 * g:].reshape(H // 128, I // 128))


def fp16_value(v: np.ndarray) -> np.ndarray:
    return v.astype(np.float16).astype(np.float32) == v


def test_generated_scales_are_fp16_values():
    for w in (FP8_SMALL_PREFILL, FP8_DSV4_DIMS_PREFILL):
        blobs = synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, np.arange(3))
        for b in range(3):
            blob = blobs[b * w.expert_bytes:(b + 1) * w.expert_bytes]
            for m in scales(blob, w.hidden, w.inter):
                assert fp16_value(m).all(), w.name


def test_shifted_scales_leave_the_fp16_grid_in_every_row_block():
    w = FP8_SMALL_PREFILL
    H, I, n = w.hidden, w.inter, 6
    blobs = synth.expert_blobs(w.seed, H, I, w.wdtype, np.arange(n))
    shifted = blobs.copy()
    shift_fp8_scales(shifted, w, n, (-6, 6, -6))
    for b in range(n):
        sl = slice(b * w.expert_bytes, (b + 1) * w.expert_bytes)
        sg, su, sd = scales(shifted[sl], H, I)
        assert (~fp16_value(sg)).any(axis=1).all()   # every Wg row block: gate/up tiles take the fp32 route
        assert (~fp16_value(sd)).any(axis=1).all()   # every Wd row block: down tiles too
        assert fp16_value(su).all()
        g0, u0, d0 = offn.dequant_blob(blobs[sl], H, I, w.wdtype)
        g1, u1, d1 = offn.dequant_blob(shifted[sl], H, I, w.wdtype)
        assert np.array_equal(g1, g0 * 2.0 ** -6)
        assert np.array_equal(u1, u0 * 2.0 ** 6)
        assert np.array_equal(d1, d0 * 2.0 ** -6)
        assert np.array_equal(shifted[sl][:3 * H * I], blobs[sl][:3 * H * I])  # the e4m3 codes are untouched


def test_one_rounding_claim_behind_the_fp16_route():
    """Every finite e4m3 value is an fp16 value, and so is a bf16 scale in
    [2^-14, 2^15] (8 significant bits); their product has at most 12
    significant bits, so rounding it once to fp16 (one fp16 multiply) gives
    what the fp32 product rounded to fp16 gives.  A bf16 scale below 2^-14
    can fall between fp16 values: rounding the scale first then differs."""
    from oracle import fp8
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)  # 0x7F / 0xFF are NaN
    w = fp8.decode_array(codes)
    assert np.array_equal(w.astype(np.float16).astype(np.float64), w)
    rng = np.random.default_rng(7)
    mant = rng.integers(0, 128, size=200)
    for exp in range(-14, 16):
        s = (1.0 + mant / 128.0) * 2.0 ** exp          # bf16 values: 1 + 7 mantissa bits
        assert np.array_equal(s.astype(np.float16).astype(np.float64), s)
        with np.errstate(over="ignore"):                 # past fp16's range both sides give inf
            prod = w[None, :] * s[:, None]               # exact in fp64
            via_f32 = (w[None, :].astype(np.float32) * s[:, None].astype(np.float32)).astype(np.float16)
            via_f16 = (w[None, :].astype(np.float16) * s[:, None].astype(np.float16))
            assert np.array_equal(prod.astype(np.float16), via_f32)
            assert np.array_equal(prod.astype(np.float16), via_f16)
    small = (1.0 + 127 / 128.0) * 2.0 ** -20             # a bf16 scale off the fp16 grid
    assert float(np.float16(small)) != small
    assert (w * small).astype(np.float16).tolist() != (w.astype(np.float16) * np.float16(small)).tolist()
