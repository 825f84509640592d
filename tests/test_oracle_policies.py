"""Comparison cache policies (oracle/policies.py) against brute force and
closed forms, then all of them against the method's global LRU on the
35B-A3B-shaped decode traces (the test prints the miss rates)."""
import numpy as np
import pytest

from oracle import policies, routing
from oracle.cache import ExpertCacheOracle
from synth import workloads as W


def _random_events(rng, L, E, k, steps):
    trace = np.stack([np.stack([rng.choice(E, size=(1, k), replace=False) for _ in range(L)])
                      for _ in range(steps)])
    return trace, policies.unique_events(trace)


def _textbook_lru_misses(events, cap):
    """One LRU list with explicit last-use stamps (no shared code with the policy)."""
    last = {}
    misses = 0
    for t, (_, experts) in enumerate(events):
        for e in experts:
            if e not in last:
                misses += 1
                if len(last) >= cap:
                    victim = min((s, x) for x, s in last.items() if x not in set(experts.tolist()))[1]
                    del last[victim]
            last[e] = t
    return misses


def test_static_split_with_one_layer_is_textbook_lru():
    rng = np.random.default_rng(3)
    _, events = _random_events(rng, 1, 12, 3, 200)
    for cap in (3, 5, 8, 12):
        m, u = policies.static_split_lru(events, 1, cap)
        assert u == 600 and m == _textbook_lru_misses(events, cap), cap


def test_static_split_shares_slots_as_stated():
    rng = np.random.default_rng(4)
    trace, events = _random_events(rng, 3, 10, 2, 50)
    # 3 layers, 7 slots: layers get 3, 2, 2; each layer alone is a textbook LRU of its share
    m, u = policies.static_split_lru(events, 3, 7)
    want = sum(_textbook_lru_misses([ev for ev in events if ev[0] == l], cap) for l, cap in enumerate((3, 2, 2)))
    assert m == want and u == 300


def test_static_layers_closed_form():
    rng = np.random.default_rng(5)
    trace, events = _random_events(rng, 4, 16, 2, 30)
    total = sum(len(x) for _, x in events)
    assert policies.static_layers(events, 4, 16, 0) == (total, total)
    assert policies.static_layers(events, 4, 16, 64) == (0, total)
    later = sum(len(x) for l, x in events if l >= 2)  # two whole layers resident
    assert policies.static_layers(events, 4, 16, 2 * 16 + 15) == (later, total)


def test_static_profile_bounds_and_monotone():
    rng = np.random.default_rng(6)
    trace, events = _random_events(rng, 2, 20, 3, 60)
    half = len(events) // 2
    after = sum(len(x) for _, x in events[half:])
    assert policies.static_profile(events, 20, 0, half) == (after, after)
    m_all, _ = policies.static_profile(events, 20, 40, half)  # every key of the profile fits
    seen = {l * 20 + int(e) for l, x in events[:half] for e in x}
    assert m_all == sum(1 for l, x in events[half:] for e in x if l * 20 + int(e) not in seen)
    ms = [policies.static_profile(events, 20, c, half)[0] for c in range(0, 41, 5)]
    assert all(a >= b for a, b in zip(ms, ms[1:]))


@pytest.mark.parametrize("w", [W.QWEN35B_DECODE, W.QWEN35B_DECODE_B4, W.QWEN35B_DECODE_B8],
                         ids=["b1-3072-slots", "b4-1740-slots", "b8-1740-slots"])
def test_policies_on_the_35b_decode_trace(w):
    """Global (layer, expert) LRU against static placements with the same
    slots on the 35B-A3B-shaped decode routing (512 steps; batch 1 with 3072
    slots, 4 and 8 streams with 1740)."""
    steps = w.steps
    logits = W.router_logits(w.replace(steps=steps))
    trace = np.stack([np.stack([routing.route(logits[s, l], w.top_k)[0] for l in range(w.num_layers)])
                      for s in range(steps)])
    events = policies.unique_events(trace)
    cache = ExpertCacheOracle(w.num_layers, w.num_experts, w.num_slots)
    for l, experts in ((l, trace[s, l]) for s in range(steps) for l in range(w.num_layers)):
        cache.event(l, experts)
    rates = {"global_lru": cache.n_miss / cache.n_unique}
    m, u = policies.static_split_lru(events, w.num_layers, w.num_slots)
    rates["static_split_lru"] = m / u
    m, u = policies.static_layers(events, w.num_layers, w.num_experts, w.num_slots)
    rates["static_layers"] = m / u
    m, u = policies.static_profile(events, w.num_experts, w.num_slots, 64 * w.num_layers)
    rates["static_profile_64_steps"] = m / u
    print(f"miss rates ({w.name}, {w.num_slots} slots, {steps} steps):", {k: round(v, 4) for k, v in rates.items()})
    # the method's cache beats placing whole layers (the offload the pages compare against)
    assert rates["global_lru"] < rates["static_layers"]


def test_previous_step_prefetch_coverage_against_a_textbook_lru():
    """k = 1 traces (the global LRU is then a textbook LRU over keys): a miss
    is covered when layer l used the same expert at the previous step and it
    was evicted since; recomputed here with an OrderedDict, on traces small
    enough that such evictions happen."""
    import collections

    from oracle import policies
    rng = np.random.default_rng(5)
    for L, E, C in ((4, 8, 3), (5, 6, 3), (6, 8, 4)):  # fewer slots than layers: last step's experts get evicted
        steps = 60
        tr = rng.integers(0, E, size=(steps, L, 1, 1)).astype(np.int32)
        misses, covered, predicted = policies.previous_step_prefetch_coverage(tr, L, E, C)
        lru = collections.OrderedDict()
        m = c = p = 0
        for s in range(steps):
            for l in range(L):
                key = l * E + int(tr[s, l, 0, 0])
                prev = l * E + int(tr[s - 1, l, 0, 0]) if s > 0 else None
                pred_missing = prev is not None and prev not in lru
                hit = key in lru
                if hit:
                    lru.move_to_end(key)
                else:
                    if len(lru) == C:
                        lru.popitem(last=False)
                    lru[key] = True
                if s > 0:
                    m += not hit
                    c += (not hit) and pred_missing and prev == key
                    p += pred_missing
        assert (misses, covered, predicted) == (m, c, p), (L, E, C)
        assert covered > 0


def test_previous_step_prefetch_covers_no_miss_on_the_decode_trace():
    """On the 35B-shaped decode routing (70% of each step's experts kept from
    the previous step) the previous step's experts are still resident when the
    next step reaches their layer, so a predictor built from them covers none
    of the misses: they are the newly drawn experts."""
    from oracle import policies
    from oracle import routing
    w = W.QWEN35B_DECODE
    steps = 40
    lg = W.router_logits(w.replace(steps=steps))
    tr = np.stack([np.stack([routing.topk(lg[s, l], w.top_k) for l in range(w.num_layers)]) for s in range(steps)])
    misses, covered, predicted = policies.previous_step_prefetch_coverage(tr, w.num_layers, w.num_experts,
                                                                          w.num_slots)
    assert misses > 0 and covered == 0 and predicted == 0


def test_frequency_prefetch_coverage_against_a_textbook_lru():
    """k = 1 traces, recomputed with an OrderedDict LRU and plain use counts:
    the predictor names the most-used non-resident experts of the layer
    (ties: lower index); a miss is covered when its expert was named."""
    import collections

    from oracle import policies
    rng = np.random.default_rng(11)
    for L, E, C, P in ((4, 8, 3, 2), (5, 6, 3, 1), (3, 10, 5, 3)):
        steps = 50
        tr = rng.integers(0, E, size=(steps, L, 1, 1)).astype(np.int32)
        got = policies.frequency_prefetch_coverage(tr, L, E, C, P, warm_steps=5)
        lru = collections.OrderedDict()
        uses = np.zeros((L, E), dtype=int)
        m = c = p = 0
        for s in range(steps):
            for l in range(L):
                order = sorted(range(E), key=lambda e: (-uses[l, e], e))
                named = [e for e in order if l * E + e not in lru][:P]
                e_now = int(tr[s, l, 0, 0])
                key = l * E + e_now
                hit = key in lru
                if hit:
                    lru.move_to_end(key)
                else:
                    if len(lru) == C:
                        lru.popitem(last=False)
                    lru[key] = True
                if s >= 5:
                    m += not hit
                    c += (not hit) and e_now in named
                    p += len(named)
                uses[l, e_now] += 1
        assert got == (m, c, p), (L, E, C, P)
        assert 0 < got[1] <= got[0]


def test_frequency_prefetch_costs_far_more_link_traffic_than_it_saves_on_the_decode_trace():
    """On the 35B-shaped decode routing the misses are fresh draws from the
    tail of each layer's expert popularity: naming the 8 most-used missing
    experts per layer covers about a tenth of the misses while copying more
    than fifty times as many blobs as it covers."""
    from oracle import policies, routing
    w = W.QWEN35B_DECODE
    steps = 48
    lg = W.router_logits(w.replace(steps=steps))
    tr = np.stack([np.stack([routing.topk(lg[s, l], w.top_k) for l in range(w.num_layers)]) for s in range(steps)])
    misses, covered, prefetched = policies.frequency_prefetch_coverage(tr, w.num_layers, w.num_experts,
                                                                       w.num_slots, 8, warm_steps=16)
    assert misses > 0 and covered < 0.25 * misses
    assert prefetched > 50 * max(covered, 1)
