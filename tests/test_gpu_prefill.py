"""Prefill layer events (T > 8 tokens) through libft against the oracle.

The prefill path groups the chunk's T*k (token, pick) rows by expert and runs
the gate/up + SwiGLU and down projections as grouped tensor-core GEMMs that
read the weights from the cache slots, then combines each token's picks.  The
routing, dedup, hit/miss and LRU decisions of the chunk are compared in full;
the FFN output on every token of a 200-token chunk (ragged against the
128-row tiles; T*k above what the route kernel groups itself) and on sampled
tokens of the full 16,384-token chunk.  Both with the next layer's fetch
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


@pytest.mark.parametrize("double_buffer", [True, False], ids=["double-buffered", "serial"])
def test_prefill_16k_chunk(double_buffer):
    from tests.harness import run_parity
    w = W.QWEN35B_PREFILL.replace(num_layers=2)
    rng = np.random.default_rng(20261202)
    tok = np.unique(np.concatenate([[0, w.tokens - 1], rng.choice(w.tokens, 10, replace=False)]))
    rep = run_parity(w, steps=1, bank_blobs=512, double_buffer=double_buffer, ffn_tokens=tok)
    assert rep["events"] == 2 and rep["ffn_checked"] == 2
    assert rep["stats"]["unique_experts"] > 300  # nearly all 256 experts per layer
    print("prefill 16k:", {k: rep[k] for k in ("max_err", "miss_rate")})
