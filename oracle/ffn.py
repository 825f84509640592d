"""Expert-blob dequantisation and the SwiGLU MoE FFN (oracle).

The pages give the expert FFN only by implication (routed experts of a
Qwen3.6-35B-A3B / DeepSeek-V4-Flash MoE layer; "FreeToken vs vLLM on one RTX
3090", "Why the performance differs").  Reading: the standard SwiGLU routed
expert of those families,

    h = silu(Wg x) * (Wu x),    silu(z) = z / (1 + exp(-z)),
    y_t = sum_j w_tj * Wd_(e_tj) h_(t, j),

computed here in fp64 with no intermediate rounding.

Blob layout (the runtime layout the host bank stores and the slots hold,
"FreeToken: Efficient Edge-Native MoE Serving ...", design paragraph: weights
pre-merged into the runtime layout): Wg [I][H], Wu [I][H], Wd [H][I]
row-major, element type f32, bf16 or fp8 e4m3.  For fp8 the three matrices
are followed by bf16 scales, one per 128 x 128 block of each matrix over its
[out][in] shape, row-block major, in the order Wg, Wu, Wd ("fp8_block",
"FreeToken: az VRAM ile büyük MoE modelleri", section "Tuzaklar"; reading: the
DeepSeek-V3-style 128 x 128 weight blocks).  A weight's value is its e4m3
value times its block's scale.
"""
from __future__ import annotations

import numpy as np

from . import fp8

W_F32, W_BF16, W_FP8 = 0, 1, 2
BLOCK = 128


def expert_bytes(hidden: int, inter: int, wdtype: int) -> int:
    n = 3 * hidden * inter
    if wdtype == W_F32:
        return 4 * n
    if wdtype == W_BF16:
        return 2 * n
    if wdtype == W_FP8:
        return n + 2 * 3 * (hidden // BLOCK) * (inter // BLOCK)
    raise ValueError(wdtype)


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dequant_blob(blob: np.ndarray, hidden: int, inter: int, wdtype: int):
    """(Wg [I,H], Wu [I,H], Wd [H,I]) in float64 from one expert blob (uint8)."""
    H, I = hidden, inter
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    assert blob.size == expert_bytes(H, I, wdtype)
    n = H * I
    if wdtype == W_F32:
        w = blob.view(np.float32).astype(np.float64)
    elif wdtype == W_BF16:
        w = _bf16_to_f64(blob.view(np.uint16))
    elif wdtype == W_FP8:
        w = fp8.decode_array(blob[:3 * n])
    else:
        raise ValueError(wdtype)
    Wg = w[0:n].reshape(I, H).copy()
    Wu = w[n:2 * n].reshape(I, H).copy()
    Wd = w[2 * n:3 * n].reshape(H, I).copy()
    if wdtype == W_FP8:
        s = _bf16_to_f64(blob[3 * n:].view(np.uint16))
        g = (I // BLOCK) * (H // BLOCK)
        for mat, scales in ((Wg, s[0:g]), (Wu, s[g:2 * g]), (Wd, s[2 * g:3 * g])):
            rows, cols = mat.shape
            grid = scales.reshape(rows // BLOCK, cols // BLOCK)
            # weight (r, c) times the scale of block (r // 128, c // 128)
            blocks = mat.reshape(rows // BLOCK, BLOCK, cols // BLOCK, BLOCK)
            blocks *= grid[:, None, :, None]
    return Wg, Wu, Wd


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def expert_ffn(x: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray) -> np.ndarray:
    """Wd (silu(Wg x) * (Wu x)) for the rows of x [n, H] -> [n, H] (float64)."""
    x = np.asarray(x, dtype=np.float64)
    g = x @ Wg.T
    u = x @ Wu.T
    return (silu(g) * u) @ Wd.T


def moe_ffn(x: np.ndarray, topk_idx: np.ndarray, gate_w: np.ndarray, weights_of) -> np.ndarray:
    """y [T, H] (float64) = sum_j w_tj * FFN_(e_tj)(x_t).

    `weights_of(e)` returns the dequantised (Wg, Wu, Wd) of expert e at this
    layer.  Each distinct expert is evaluated once on the tokens that chose it.
    """
    x = np.asarray(x, dtype=np.float64)
    topk_idx = np.asarray(topk_idx)
    gate_w = np.asarray(gate_w, dtype=np.float64)
    y = np.zeros_like(x)
    for e in sorted({int(v) for v in topk_idx.ravel()}):
        tok, j = np.nonzero(topk_idx == e)
        out = expert_ffn(x[tok], *weights_of(e))
        y[tok] += gate_w[tok, j][:, None] * out
    return y
