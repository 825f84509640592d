"""Checks of the shared input generators (not of the method)."""
import numpy as np

import synth
from synth import workloads as W


def test_bf16_encoder_is_round_to_nearest_even():
    x = synth.normal(synth.key(1), 20000) * np.float32(3.0)
    bits = synth.bf16_bits(x)
    v = synth.bf16_values(bits).astype(np.float64)
    up = synth.bf16_values(bits + 1).astype(np.float64)
    dn = synth.bf16_values(bits - 1).astype(np.float64)
    xd = x.astype(np.float64)
    err = np.abs(v - xd)
    assert np.all(err <= np.abs(up - xd)) and np.all(err <= np.abs(dn - xd))


def test_generators_are_deterministic_and_thread_independent(monkeypatch):
    a = synth.expert_blobs(5, 128, 128, synth.W_FP8, [3, 9])
    monkeypatch.setattr(synth, "threads", lambda: 1)
    b = synth.expert_blobs(5, 128, 128, synth.W_FP8, [3, 9])
    np.testing.assert_array_equal(a, b)
    c = synth.expert_blobs(5, 128, 128, synth.W_FP8, [9])
    np.testing.assert_array_equal(a[a.size // 2:], c)


def test_correlated_routing_keeps_about_70_percent():
    lg = synth.router_decode(W.QWEN35B_DECODE.seed, 0, 4, 256, 8, 200)
    top = np.argsort(-lg, axis=-1)[..., :8]
    ov = [len(set(top[s, l]) & set(top[s - 1, l])) / 8 for s in range(1, 200) for l in range(4)]
    assert 0.66 < np.mean(ov) < 0.80
    # the lifted experts are the top-8 by a wide margin
    srt = np.sort(lg, axis=-1)
    assert np.all(srt[1:, :, -8] - srt[1:, :, -9] > 5)


def test_workload_sizes():
    assert W.QWEN35B_DECODE.expert_bytes == 6291456
    assert W.DSV4_DECODE.expert_bytes == 25168896
    assert W.TINY.expert_bytes == 393216
    assert (W.DSV4_DECODE.num_slots, W.DSV4_DECODE.resize_slots) == (2383, 1191)
