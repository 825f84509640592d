"""Prefill layer events (T > 8 tokens) through libft against the oracle.

The prefill path groups the chunk's T*k (token, pick) rows by expert and runs
the gate/up + SwiGLU and down projections as grouped tcgen05 GEMMs that read
the weights from the cache slots, then combines each token's picks.  The
routing, dedup, hit/miss and LRU decisions of the chunk are compared in full.
The FFN output is compared on every token of a 200-token chunk (ragged
against the 128-row tiles; T*k above what the route kernel groups itself),
and on the full 16,384-token chunk: every row of its first layer, and on the
second layer 512 seeded tokens plus every token that picked the layer's
rarest expert (the expert with the fewest rows, whose single ragged tile is
the likeliest to be mishandled).  Both with the next layer's fetch
double-buffered and without.
"""
import numpy as np
import pytest

from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("double_buffer", [True, False], ids=["double-buffered", "serial"])
def test_prefill_chunk_full_parity(double_buffer):
    from tests.harness import run_parity
    w = W.QWEN35B_PREFILL.replace(num_layers=2, tokens=200)
    rep = run_parity(w, steps=1, bank_blobs=512, double_buffer=double_buffer)
    assert rep["events"] == 2 and rep["ffn_checked"] == 2 and rep["slots_checked"] > 0
    print("prefill 200:", {k: rep[k] for k in ("max_err", "miss_rate")})


def sampled_tokens(layer, idx, T=W.QWEN35B_PREFILL.tokens):
    """Layer 0: every token.  Other layers: 512 seeded tokens plus every token
    whose top-k holds the rarest unique expert."""
    if layer == 0:
        return None
    experts, counts = np.unique(idx, return_counts=True)
    rare = experts[np.argmin(counts)]
    rng = np.random.default_rng(20261202 + layer)
    tok = rng.choice(T, 512, replace=False)
    tok = np.union1d(tok, np.flatnonzero((idx == rare).any(axis=1)))
    return np.union1d(tok, [0, T - 1])


@pytest.mark.parametrize("double_buffer", [True, False], ids=["double-buffered", "serial"])
def test_prefill_16k_chunk(double_buffer):
    from tests.harness import run_parity
    w = W.QWEN35B_PREFILL.replace(num_layers=2)
    rep = run_parity(w, steps=1, bank_blobs=512, double_buffer=double_buffer, ffn_tokens=sampled_tokens)
    assert rep["events"] == 2 and rep["ffn_checked"] == 2
    assert rep["stats"]["unique_experts"] > 300  # nearly all 256 experts per layer
    print("prefill 16k:", {k: rep[k] for k in ("max_err", "max_rms_err", "miss_rate")})


# fp8 e4m3 experts with bf16 128 x 128 block scales on the prefill path: the
# weights are dequantised to fp16 (times their block's scale) in shared memory
# and multiplied with fp16 activations on the tensor cores.  A small shape (ragged tiles, 64 experts)
# and the DeepSeek-V4-Flash-shaped layer dimensions (hidden 4096,
# intermediate 2048) with 32 experts so the fp64 oracle stays quick.
FP8_SMALL_PREFILL = W.DSV4_DECODE.replace(name="fp8-prefill-1024x512", num_layers=2, num_experts=64, hidden=1024,
                                          inter=512, tokens=300, steps=1, num_slots=256, routing=W.ROUTE_ZIPF_IID,
                                          resize_step=-1, bank_blobs=0)
FP8_DSV4_DIMS_PREFILL = W.DSV4_DECODE.replace(name="fp8-prefill-dsv4-dims", num_layers=2, num_experts=32,
                                              tokens=256, steps=1, num_slots=64, routing=W.ROUTE_ZIPF_IID,
                                              resize_step=-1, bank_blobs=0)


@pytest.mark.parametrize("w", [FP8_SMALL_PREFILL, FP8_DSV4_DIMS_PREFILL], ids=["1024x512", "dsv4-dims"])
def test_fp8_prefill_parity(w):
    from tests.harness import run_parity
    rep = run_parity(w, steps=1, double_buffer=True)
    assert rep["events"] == 2 and rep["ffn_checked"] == 2 and rep["slots_checked"] > 0
    print("fp8 prefill:", {k: rep[k] for k in ("max_err", "max_rms_err", "miss_rate")})


def test_fp8_prefill_parity_scales_off_fp16():
    # Wg and Wd block scales times 2^-6 (Wu times 2^6 keeps h at its usual size):
    # every Wg and Wd row block then has a scale that is not an fp16 value, so
    # every tile of both GEMMs dequantises through the fp32 product instead of
    # the fp16 multiply the generated scales allow (tests/test_fp8_scale_fixture.py)
    from tests.harness import run_parity
    rep = run_parity(FP8_SMALL_PREFILL, steps=1, double_buffer=True, fp8_scale_shifts=(-6, 6, -6))
    assert rep["events"] == 2 and rep["ffn_checked"] == 2
    print("fp8 prefill, scales off the fp16 grid:", {k: rep[k] for k in ("max_err", "max_rms_err")})
