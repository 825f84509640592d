"""Pins of the oracle's expert dequantisation and SwiGLU MoE FFN.

* closed forms on hand-built experts (identity / permutation matrices) whose
  outputs are computed here from math.exp, so a swapped gate/up matrix, a
  transposed down matrix, a wrong silu or a gate weight on the wrong expert
  gives a different number;
* the blob layout read back from hand-packed blobs;
* the dense identity: evaluating every expert of the layer with zero gates
  except the selected ones gives the same y;
* fp8 block scales applied to the right 128 x 128 blocks.
"""
import math

import numpy as np
import pytest

import synth
from oracle import ffn, fp8


def pack_blob(Wg, Wu, Wd, wdtype):
    parts = [np.asarray(Wg), np.asarray(Wu), np.asarray(Wd)]
    if wdtype == ffn.W_F32:
        return np.concatenate([p.astype(np.float32).ravel() for p in parts]).view(np.uint8)
    if wdtype == ffn.W_BF16:
        return np.concatenate([synth.bf16_bits(p.astype(np.float32)).ravel() for p in parts]).view(np.uint8)
    raise ValueError


def silu(z):
    return z / (1.0 + math.exp(-z))


def test_silu_closed_forms():
    z = np.array([0.0, 30.0, -30.0, 1.0, -2.0])
    s = ffn.silu(z)
    assert s[0] == 0.0
    assert abs(s[1] - 30.0) < 1e-11 and abs(s[2]) < 1e-11
    assert abs(s[3] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(s[4] - (-2.0 / (1.0 + math.exp(2.0)))) < 1e-16
    # silu(x) - silu(-x) = x
    x = np.linspace(-5, 5, 101)
    np.testing.assert_allclose(ffn.silu(x) - ffn.silu(-x), x, atol=1e-14)


@pytest.mark.parametrize("wdtype", [ffn.W_F32, ffn.W_BF16])
def test_single_expert_closed_form(wdtype):
    # H = I = 2: Wg = 2*Id, Wu = Id, Wd = swap permutation
    Wg = np.array([[2.0, 0.0], [0.0, 2.0]])
    Wu = np.eye(2)
    Wd = np.array([[0.0, 1.0], [1.0, 0.0]])
    blob = pack_blob(Wg, Wu, Wd, wdtype)
    g, u, d = ffn.dequant_blob(blob, 2, 2, wdtype)
    np.testing.assert_array_equal(g, Wg)
    np.testing.assert_array_equal(d, Wd)
    x = np.array([[1.0, -2.0]])
    y = ffn.moe_ffn(x, np.array([[0]]), np.array([[1.0]]), lambda e: (g, u, d))
    h = [silu(2.0) * 1.0, silu(-4.0) * -2.0]
    assert abs(y[0, 0] - h[1]) < 1e-15 and abs(y[0, 1] - h[0]) < 1e-15


def test_gate_weights_go_to_their_own_expert():
    H = I = 2
    e0 = (np.eye(2) * 2, np.eye(2), np.eye(2))              # h = silu(2x) * x
    e1 = (np.eye(2), np.eye(2) * 3, np.eye(2))              # h = silu(x) * 3x
    experts = {0: e0, 1: e1}
    x = np.array([[0.5, -1.5], [1.0, 2.0]])
    idx = np.array([[1, 0], [0, 1]])
    w = np.array([[0.7, 0.3], [0.6, 0.4]])
    y = ffn.moe_ffn(x, idx, w, lambda e: experts[e])
    for t in range(2):
        for c in range(H):
            v = x[t, c]
            f0 = silu(2 * v) * v
            f1 = silu(v) * 3 * v
            want = sum(w[t, j] * (f0 if idx[t, j] == 0 else f1) for j in range(2))
            assert abs(y[t, c] - want) < 1e-14


@pytest.mark.parametrize("wdtype", [ffn.W_F32, ffn.W_BF16])
def test_blob_layout_order(wdtype):
    H, I = 8, 4
    rng = np.random.default_rng(0)
    Wg = rng.integers(-8, 8, (I, H)) / 8.0
    Wu = rng.integers(-8, 8, (I, H)) / 16.0
    Wd = rng.integers(-8, 8, (H, I)) / 32.0
    g, u, d = ffn.dequant_blob(pack_blob(Wg, Wu, Wd, wdtype), H, I, wdtype)
    np.testing.assert_array_equal(g, Wg)
    np.testing.assert_array_equal(u, Wu)
    np.testing.assert_array_equal(d, Wd)


def test_fp8_block_scales_applied_per_block():
    H, I = 256, 128
    n = H * I
    codes = np.full(3 * n, 0x38, dtype=np.uint8)          # every weight = 1.0 before scaling
    # scale grids: Wg, Wu [1 x 2] blocks, Wd [2 x 1] blocks
    scales = np.array([1.0, 2.0, 4.0, 8.0, 0.5, 0.25], dtype=np.float32)
    blob = np.concatenate([codes, synth.bf16_bits(scales).view(np.uint8)])
    assert blob.size == ffn.expert_bytes(H, I, ffn.W_FP8)
    g, u, d = ffn.dequant_blob(blob, H, I, ffn.W_FP8)
    assert np.all(g[:, :128] == 1.0) and np.all(g[:, 128:] == 2.0)
    assert np.all(u[:, :128] == 4.0) and np.all(u[:, 128:] == 8.0)
    assert np.all(d[:128, :] == 0.5) and np.all(d[128:, :] == 0.25)


def test_fp8_scale_grid_is_row_block_major_on_a_non_square_grid():
    """H = 384, I = 256: Wg and Wu have 2 x 3 grids of 128 x 128 blocks, Wd a
    3 x 2 grid; every block gets its own scale and every weight its own code.
    Each weight must equal its code's E4M3 value times the scale of block
    (r // 128, c // 128) taken from the matrix's grid in row-block-major order,
    the format the blob layout states.  A transposed (column-block-major) grid
    puts other scales on 4 of the 6 blocks of each matrix, so it fails here."""
    H, I = 384, 256
    n = H * I
    codes = np.empty(3 * n, dtype=np.uint8)
    # finite codes only (0x00..0x7e, then the same with the sign bit), varied per element
    codes[:] = (np.arange(3 * n) * 37) % 0x7F
    codes[1::5] |= 0x80
    grid_g = (I // 128) * (H // 128)                 # 6 blocks each for Wg, Wu, Wd
    scales = np.array([2.0 ** (j - 9) for j in range(3 * grid_g)], dtype=np.float32)  # all distinct, exact in bf16
    blob = np.concatenate([codes, synth.bf16_bits(scales).view(np.uint8)])
    assert blob.size == ffn.expert_bytes(H, I, ffn.W_FP8)
    g, u, d = ffn.dequant_blob(blob, H, I, ffn.W_FP8)
    mats = ((g, I, H, 0), (u, I, H, grid_g), (d, H, I, 2 * grid_g))
    for m, (mat, rows, cols, s0) in enumerate(mats):
        col_blocks = cols // 128
        for r in range(rows):
            for c in range(0, cols, 7):          # every 7th column of every row: all blocks, many codes
                code = int(codes[m * n + r * cols + c])
                want = fp8.decode(code) * float(scales[s0 + (r // 128) * col_blocks + c // 128])
                assert mat[r, c] == want, (m, r, c)


@pytest.mark.parametrize("wdtype,H,I", [(ffn.W_F32, 64, 32), (ffn.W_BF16, 128, 64), (ffn.W_FP8, 256, 128)])
def test_dense_identity_all_experts_zero_gates(wdtype, H, I):
    E, k, T = 8, 2, 6
    blobs = synth.expert_blobs(3, H, I, wdtype, list(range(E))).reshape(E, -1)
    W = [ffn.dequant_blob(blobs[e], H, I, wdtype) for e in range(E)]
    x = synth.normal(synth.key(4, H), T * H).reshape(T, H)
    lg = synth.normal(synth.key(5, E), T * E).reshape(T, E)
    from oracle import routing
    idx, w = routing.route(lg, k)
    y = ffn.moe_ffn(x, idx, w, lambda e: W[e])
    dense = np.zeros((T, E))
    for t in range(T):
        dense[t, idx[t]] = w[t]
    yd = sum(dense[:, e:e + 1] * ffn.expert_ffn(x, *W[e]) for e in range(E))
    np.testing.assert_allclose(y, yd, rtol=1e-12, atol=1e-14)


def test_generated_bf16_weights_decode_to_generator_values():
    H, I = 64, 32
    blob = synth.expert_blobs(8, H, I, ffn.W_BF16, [5])
    g, u, d = ffn.dequant_blob(blob, H, I, ffn.W_BF16)
    raw = synth.bf16_values(blob.view(np.uint16)).astype(np.float64)
    np.testing.assert_array_equal(g.ravel(), raw[:H * I])
    np.testing.assert_array_equal(d.ravel(), raw[2 * H * I:])
    assert 0.015 < raw.std() < 0.025


def test_generated_fp8_blob_dequantises_close_to_unquantised_weights():
    # generator stores q = e4m3(w / s) with s = bf16(max|w| / 448): |w - q*s| <= s * 2^-4 * |q|-ish
    H, I = 256, 128
    f32 = synth.expert_blobs(9, H, I, ffn.W_F32, [2]).view(np.float32).astype(np.float64)
    g, u, d = ffn.dequant_blob(synth.expert_blobs(9, H, I, ffn.W_FP8, [2]), H, I, ffn.W_FP8)
    deq = np.concatenate([g.ravel(), u.ravel(), d.ravel()])
    rel = np.abs(deq - f32) / np.maximum(np.abs(f32), 1e-3)
    assert np.median(rel) < 0.04 and np.max(np.abs(deq - f32)) < 0.01
    assert np.isfinite(fp8.TABLE[:0x7F]).all()
