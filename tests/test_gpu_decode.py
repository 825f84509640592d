"""GPU parity of the decode path through the C ABI against the CPU oracle.

Decisions (top-k indices, unique set, hit flags, victims, evicted keys, slot
tables, counters) must be bit-exact at every event; FFN outputs within
max|diff| <= tol * RMS(ref) per layer event (1e-4 for fp32, 2e-2 for
bf16/fp8); gates within 2e-6.  The fetched slots must hold their blob's bytes.
"""
import pytest
import torch

import synth
from synth import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from tests.harness import run_parity


@pytest.mark.parametrize("fetch_mode", [0, 1])
@pytest.mark.parametrize("double_buffer", [True, False])
def test_tiny_full_parity(fetch_mode, double_buffer):
    rep = run_parity(W.TINY, fetch_mode=fetch_mode, double_buffer=double_buffer)
    assert rep["events"] == 128 and rep["ffn_checked"] == 128
    assert rep["max_err"] <= 1e-4


def test_tiny_two_copy_streams():
    rep = run_parity(W.TINY, fetch_mode=0, copy_streams=2, steps=32)
    assert rep["events"] == 64


def test_tiny_tie_heavy_logits():
    w = W.TINY
    lg = synth.router_ties(w.seed, 3, (64, w.num_layers, w.tokens, w.num_experts))
    rep = run_parity(w, logits=lg)
    assert rep["events"] == 128


def test_qwen35b_decode_full_512_steps():
    """Full 512-step decode decision stream at the 35B-A3B shape (aliased 1024-blob bank)."""
    rep = run_parity(W.QWEN35B_DECODE, bank_blobs=1024, check_tables_every=41, ffn_every=53)
    assert rep["events"] == 512 * 40
    print("qwen35b decode:", rep)


def test_qwen35b_decode_copy_engine_mode():
    rep = run_parity(W.QWEN35B_DECODE, steps=48, fetch_mode=0, bank_blobs=512, check_tables_every=7, ffn_every=5)
    assert rep["events"] == 48 * 40


@pytest.mark.parametrize("w", [W.QWEN35B_DECODE_B4, W.QWEN35B_DECODE_B8], ids=["b4", "b8"])
def test_qwen35b_multistream(w):
    rep = run_parity(w, steps=96, bank_blobs=1024, check_tables_every=13, ffn_every=7)
    assert rep["events"] == 96 * 40


def test_dsv4_fp8_with_resize():
    """fp8 block-scaled experts, 1024 steps, shrink 2383 -> 1191 slots before
    step 512.  Every 61st layer event's FFN (403 events, about 2 s of oracle
    time each) is checked by a pool of host worker processes while the GPU
    run continues."""
    w = W.DSV4_DECODE
    rep = run_parity(w, check_tables_every=97, ffn_every=61, ffn_workers=12)
    assert rep["events"] == 1024 * 24 and rep["resize_moves"] > 0
    assert rep["ffn_checked"] == len(range(0, 1024 * 24, 61))
    print("dsv4:", rep)


@pytest.mark.parametrize("fetch_mode", [0, 1])
@pytest.mark.parametrize("double_buffer", [True, False])
def test_tiny_step_graph_replay(double_buffer, fetch_mode):
    from tests.harness import run_parity_graph
    rep = run_parity_graph(W.TINY, steps=64, double_buffer=double_buffer, fetch_mode=fetch_mode)
    assert rep["events"] == 128 and rep["ffn_checked"] == 128


@pytest.mark.parametrize("fetch_mode", [0, 1])
def test_qwen35b_step_graph_replay(fetch_mode):
    from tests.harness import run_parity_graph
    rep = run_parity_graph(W.QWEN35B_DECODE, steps=40, bank_blobs=512, ffn_every=13, fetch_mode=fetch_mode)
    assert rep["events"] == 40 * 40


@pytest.mark.parametrize("w", [W.QWEN35B_DECODE_B4, W.QWEN35B_DECODE_B8], ids=["b4", "b8"])
def test_qwen35b_multistream_step_graph_replay(w):
    """4 and 8 decode streams sharing the 1740-slot cache, replayed through a
    captured step graph (routing of every layer runs ahead of the FFNs, each
    fetch inside the FFN kernel before it) against the oracle."""
    from tests.harness import run_parity_graph
    rep = run_parity_graph(w, steps=48, bank_blobs=1024, ffn_every=7)
    assert rep["events"] == 48 * 40 and rep["ffn_checked"] > 0


@pytest.mark.parametrize("fetch_mode", [0, 1])
def test_qwen35b_timing_graph_keeps_dependencies(fetch_mode):
    """A graph with timing event nodes computes the same results, and each
    layer's FFN starts after its route (and, in SM-pull mode, its fetch) has
    ended.  In copy-engine mode the graph holds no fetch events: the trace
    marks them -1 and the per-layer fetch times are 0."""
    from tests.harness import run_parity_graph
    rep = run_parity_graph(W.QWEN35B_DECODE, steps=6, bank_blobs=512, ffn_every=3, timing=True,
                           fetch_mode=fetch_mode)
    tr = rep["trace"]  # [L][route b/e, fetch b/e, ffn b/e]
    route_ms, fetch_ms, ffn_ms, step_ms = rep["timing"]
    print("trace (us):", (1e3 * tr[:6]).round(1).tolist())
    assert step_ms > 0 and (route_ms > 0).all() and (ffn_ms > 0).all()
    for l in range(tr.shape[0]):
        assert tr[l, 1] <= tr[l, 4], l
        if fetch_mode == 1:
            assert tr[l, 3] <= tr[l, 4], l
        else:
            assert tr[l, 2] == -1.0 and tr[l, 3] == -1.0 and fetch_ms[l] == 0.0, l
