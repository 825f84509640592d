"""Pins of the oracle's global LRU expert cache.

* k = 1 traces against a textbook LRU written here on an OrderedDict (no slots):
  with one key per event every last-use time is distinct, so the LRU order is
  total and hit/miss and the evicted key are unique.
* k > 1 traces against a brute-force slot cache that picks each victim by a
  linear scan for the minimum (last-use, slot) - selection, not sorting.
* slot-table invariants after every event, the compulsory-miss case, the
  capacity error when the pin rule binds, and the resize definition.
"""
import collections
import itertools

import numpy as np
import pytest

import synth
from oracle import routing
from oracle.cache import CapacityError, ExpertCacheOracle


def random_trace(seed, L, E, k, T, steps, ties=False):
    if ties:
        lg = synth.router_ties(seed, 0, (steps, L, T, E))
    else:
        lg = synth.normal(synth.key(seed, L, E, k), steps * L * T * E).reshape(steps, L, T, E)
    return [[routing.topk(lg[s, l], k) for l in range(L)] for s in range(steps)]


def check_invariants(c: ExpertCacheOracle, ev, prev_slots):
    occ = np.flatnonzero(c.slot_key >= 0)
    assert len(occ) <= c.C
    # bijection between occupied slots and present keys
    present = np.flatnonzero(c.key_to_slot >= 0)
    assert len(present) == len(occ)
    for s in occ:
        assert c.key_to_slot[c.slot_key[s]] == s
    for key in present:
        assert c.slot_key[c.key_to_slot[key]] == key
    # hits + misses = unique
    assert int(ev.hit.sum()) + len(ev.miss_expert) == len(ev.unique)
    # no victim among this event's hit slots or the previous event's slots
    hit_slots = set(ev.unique_slot[ev.hit.astype(bool)].tolist())
    for s in ev.miss_slot.tolist():
        assert s not in hit_slots and s not in prev_slots
    # every unique expert present with last-use = t
    for e, s in zip(ev.unique.tolist(), ev.unique_slot.tolist()):
        assert c.key_to_slot[ev.layer * c.E + e] == s
        assert c.slot_ts[s] == ev.t


@pytest.mark.parametrize("L,E,C,seed", [(1, 4, 2, 1), (2, 8, 3, 2), (3, 8, 5, 3), (6, 8, 20, 4), (2, 16, 7, 5)])
def test_k1_matches_textbook_lru(L, E, C, seed):
    trace = random_trace(seed, L, E, 1, 1, 300)
    c = ExpertCacheOracle(L, E, C)
    lru = collections.OrderedDict()
    for s in range(300):
        for l in range(L):
            key = l * E + int(trace[s][l][0, 0])
            ev = c.event(l, trace[s][l])
            if key in lru:
                lru.move_to_end(key)
                assert ev.hit.tolist() == [1]
            else:
                assert ev.hit.tolist() == [0]
                evicted = -1
                if len(lru) == C:
                    evicted, _ = lru.popitem(last=False)
                lru[key] = True
                assert ev.evicted_key.tolist() == [evicted]
    assert set(lru) == set(np.flatnonzero(c.key_to_slot >= 0).tolist())


class BruteSlotCache:
    """Same definition, different algorithm: victims chosen one by one by a linear scan."""

    def __init__(self, L, E, C):
        self.E, self.C = E, C
        self.key = [-1] * C
        self.ts = [-1] * C
        self.t = 0
        self.prev = set()

    def event(self, layer, idx):
        U = sorted(set(int(v) for v in idx.ravel()))
        where = {k: s for s, k in enumerate(self.key) if k >= 0}
        hit_slots = {where[layer * self.E + e] for e in U if layer * self.E + e in where}
        misses = [e for e in U if layer * self.E + e not in where]
        chosen, evicted = [], []
        for e in misses:
            best = None
            for s in range(self.C):
                if s in hit_slots or s in self.prev or s in chosen:
                    continue
                if best is None or (self.ts[s], s) < (self.ts[best], best):
                    best = s
            if best is None:
                raise CapacityError("brute")
            chosen.append(best)
            evicted.append(self.key[best])
            self.key[best] = layer * self.E + e
        slots = []
        for e in U:
            s = self.key.index(layer * self.E + e)
            self.ts[s] = self.t
            slots.append(s)
        self.prev = set(slots)
        self.t += 1
        return U, misses, chosen, evicted, slots


@pytest.mark.parametrize("L,E,k,T,C,ties,seed", [
    (2, 16, 2, 1, 12, False, 7), (2, 16, 2, 1, 4, False, 8), (3, 8, 3, 2, 14, True, 9),
    (4, 8, 2, 3, 12, True, 10), (6, 8, 4, 1, 20, False, 11), (1, 16, 4, 4, 32, True, 12),
])
def test_k_gt1_matches_brute_force_slot_scan(L, E, k, T, C, ties, seed):
    trace = random_trace(seed, L, E, k, T, 80, ties)
    c, b = ExpertCacheOracle(L, E, C), BruteSlotCache(L, E, C)
    prev_slots = set()
    for s in range(80):
        for l in range(L):
            ev = c.event(l, trace[s][l])
            U, misses, chosen, evicted, slots = b.event(l, trace[s][l])
            assert ev.unique.tolist() == U
            assert ev.miss_expert.tolist() == misses
            assert ev.miss_slot.tolist() == chosen
            assert ev.evicted_key.tolist() == evicted
            assert ev.unique_slot.tolist() == slots
            check_invariants(c, ev, prev_slots)
            prev_slots = set(slots)
    assert c.slot_key.tolist() == b.key and c.slot_ts.tolist() == b.ts


def test_compulsory_misses_only_when_cache_holds_everything():
    L, E, k = 3, 16, 2
    trace = random_trace(21, L, E, k, 2, 50)
    c = ExpertCacheOracle(L, E, L * E)
    seen = set()
    for s in range(50):
        for l in range(L):
            ev = c.event(l, trace[s][l])
            keys = {l * E + int(e) for e in ev.unique}
            assert {l * E + int(e) for e in ev.miss_expert} == keys - seen
            assert ev.evicted_key.tolist() == [-1] * len(ev.miss_expert)
            seen |= keys
    assert c.n_miss == len(seen) and c.n_evict == 0


def test_cold_cache_fills_slots_in_order():
    c = ExpertCacheOracle(2, 8, 10)
    ev = c.event(0, np.array([[5, 1, 3]]))
    assert ev.unique.tolist() == [1, 3, 5] and ev.miss_slot.tolist() == [0, 1, 2]
    ev = c.event(1, np.array([[0, 7]]))
    assert ev.miss_slot.tolist() == [3, 4]


def test_pin_rule_binds_and_raises_capacity_error():
    c = ExpertCacheOracle(1, 8, 6)
    c.event(0, np.array([[0, 1, 2, 3]]))
    # the previous event's 4 slots are pinned: 2 candidates for 4 misses
    with pytest.raises(CapacityError):
        c.event(0, np.array([[4, 5, 6, 7]]))


def test_pin_rule_excludes_previous_event_slots():
    c = ExpertCacheOracle(2, 8, 4)
    c.event(0, np.array([[0, 1]]))      # slots 0,1 (t=0)
    c.event(1, np.array([[0, 1]]))      # slots 2,3 (t=1), pins 0,1? no: pins event-0 slots
    ev = c.event(0, np.array([[2, 3]]))  # t=2: pinned = slots 2,3; LRU = slots 0,1 -> both evicted
    assert ev.miss_slot.tolist() == [0, 1] and ev.evicted_key.tolist() == [0, 1]
    ev = c.event(1, np.array([[5]]))     # t=3: pinned = 0,1; candidates 2,3 (ts 1) -> slot 2
    assert ev.miss_slot.tolist() == [2] and ev.evicted_key.tolist() == [8 + 0]


@pytest.mark.parametrize("new_C", [3, 6, 9, 12, 16])
def test_resize_keeps_most_recent_and_compacts(new_C):
    L, E, k, C = 4, 16, 2, 12
    trace = random_trace(31, L, E, k, 1, 40)
    c = ExpertCacheOracle(L, E, C)
    for s in range(40):
        for l in range(L):
            c.event(l, trace[s][l])
    before = {int(c.slot_key[s]): (int(c.slot_ts[s]), s) for s in range(C) if c.slot_key[s] >= 0}
    # expected survivors: the keys LRU would evict last (drop the first in (ts, slot) order)
    order = sorted(before, key=lambda key: before[key])
    survivors = set(order[max(0, len(order) - new_C):])
    moves = c.resize(new_C)
    assert c.C == new_C and len(c.slot_key) == new_C
    after = {int(c.slot_key[s]): s for s in range(new_C) if c.slot_key[s] >= 0}
    assert set(after) == survivors
    for key, s in after.items():
        assert c.slot_ts[s] == before[key][0]          # last-use kept
        assert c.key_to_slot[key] == s
        if before[key][1] < new_C:
            assert s == before[key][1]                  # survivors below C' stay put
    assert np.count_nonzero(c.key_to_slot >= 0) == len(survivors)
    # movers: ascending old slot -> ascending lowest free slots
    assert [m[0] for m in moves] == sorted(m[0] for m in moves)
    stay = {before[key][1] for key in survivors if before[key][1] < new_C}
    free = [s for s in range(new_C) if s not in stay]
    assert [m[1] for m in moves] == free[:len(moves)]
    assert all(c.slot_key[new] == key for key in survivors for (old, new) in moves if before[key][1] == old)
    # the next event has no t-1 pin: with everything full it may evict any non-hit slot
    ev = c.event(0, trace[0][0])
    assert int(ev.hit.sum()) + len(ev.miss_expert) == len(ev.unique)


@pytest.mark.parametrize("L,E,C,new_C,seed", [(2, 8, 9, 4, 41), (3, 8, 12, 5, 42), (4, 16, 20, 7, 43),
                                               (2, 16, 6, 10, 44), (1, 4, 3, 2, 45)])
def test_resize_k1_matches_textbook_lru_at_the_new_capacity(L, E, C, new_C, seed):
    """k = 1: one key per event, so every resident key has its own last-use
    time and LRU order is total.  After resize(C') the resident keys must be
    exactly the C' most recently used keys of a textbook OrderedDict LRU, and
    the next 100 events must hit, miss and evict exactly as that LRU does at
    capacity C' (no slot arithmetic involved)."""
    trace = random_trace(seed, L, E, 1, 1, 160)
    c = ExpertCacheOracle(L, E, C)
    lru = collections.OrderedDict()

    def access(key, cap):
        if key in lru:
            lru.move_to_end(key)
            return True, -1
        ev = lru.popitem(last=False)[0] if len(lru) == cap else -1
        lru[key] = True
        return False, ev

    for s in range(60):
        for l in range(L):
            c.event(l, trace[s][l])
            access(l * E + int(trace[s][l][0, 0]), C)
    c.resize(new_C)
    while len(lru) > new_C:
        lru.popitem(last=False)
    assert set(np.flatnonzero(c.key_to_slot >= 0).tolist()) == set(lru)
    n = 0
    for s in range(60, 160):
        for l in range(L):
            key = l * E + int(trace[s][l][0, 0])
            ev = c.event(l, trace[s][l])
            hit, evicted = access(key, new_C)
            assert ev.hit.tolist() == [int(hit)], (s, l)
            assert ev.evicted_key.tolist() == ([] if hit else [evicted]), (s, l)
            n += 1
            if n == 100:
                assert set(np.flatnonzero(c.key_to_slot >= 0).tolist()) == set(lru)
                return


@pytest.mark.parametrize("new_C", [4, 7, 10])
def test_resize_drops_the_keys_the_next_misses_would_evict(new_C):
    """Ties in last use (k = 3 picks per event share one time): shrinking
    drops exactly the keys that the victim rule of an event would evict
    first.  The same cache state is shrunk in one copy and, in another,
    served one event of never-seen experts on a layer whose misses need
    exactly that many victims with no pin (the first event after a resize
    pins nothing, so a same-size resize clears the pin first).  Flipping the
    tie order of either rule (slot descending among equal last use) changes
    the dropped set and fails here."""
    import copy
    L, E, k, C = 3, 32, 3, 12
    trace = random_trace(51, L, E, k, 1, 30, ties=True)
    base = ExpertCacheOracle(L + 1, E, C)
    for s in range(30):
        for l in range(L):
            base.event(l, trace[s][l])
    occupied = int(np.count_nonzero(base.slot_key >= 0))
    n_drop = occupied - new_C
    assert n_drop > 0
    shrunk = copy.deepcopy(base)
    before = {int(k_) for k_ in shrunk.slot_key if k_ >= 0}
    shrunk.resize(new_C)
    dropped = before - {int(k_) for k_ in shrunk.slot_key if k_ >= 0}
    evictor = copy.deepcopy(base)
    evictor.resize(C)                                       # same size: only clears the pin
    ev = evictor.event(L, np.arange(n_drop, dtype=np.int32)[None, :])   # layer L: all misses
    assert set(ev.evicted_key.tolist()) == dropped and len(dropped) == n_drop


def test_miss_rate_counts_unique_experts_per_event():
    c = ExpertCacheOracle(1, 8, 8)
    c.event(0, np.array([[1, 2], [2, 3]]))   # U = {1,2,3}: 3 misses
    c.event(0, np.array([[1, 4], [4, 1]]))   # U = {1,4}: 1 hit, 1 miss
    assert (c.n_unique, c.n_hit, c.n_miss) == (5, 1, 4)
    assert c.miss_rate() == 4 / 5


def test_exhaustive_tiny_traces_match_brute_force():
    # every length-4 trace of single-token top-2 picks over 4 experts, one layer, 3..5 slots
    pairs = [np.array([list(p)]) for p in itertools.permutations(range(4), 2)]
    for C in (4, 5):
        for tr in itertools.product(pairs, repeat=3):
            c, b = ExpertCacheOracle(1, 4, C), BruteSlotCache(1, 4, C)
            for idx in tr:
                ev = c.event(0, idx)
                _, _, chosen, evicted, slots = b.event(0, idx)
                assert ev.miss_slot.tolist() == chosen and ev.unique_slot.tolist() == slots
                assert ev.evicted_key.tolist() == evicted


def test_tables_are_consistent_with_the_event_records():
    """tables() (what the GPU tables are compared with) against the events:
    key_to_slot and slot_key are inverse maps over the resident keys, no more
    than C keys are resident, and each slot's last use is the last event that
    put its key there or hit it (recomputed from the event records)."""
    import numpy as _np
    from oracle.cache import ExpertCacheOracle as _C
    rng = _np.random.default_rng(11)
    L, E, k, C = 3, 12, 3, 12  # C = 2 * min(T*k, E): the capacity bound
    cache = _C(L, E, C)
    last_use = {}
    for t in range(120):
        l = t % L
        ev = cache.event(l, rng.choice(E, size=(2, k), replace=True))
        for u, e in enumerate(ev.unique.tolist()):
            last_use[int(ev.unique_slot[u])] = (l * E + e, ev.t)
        k2s, sk, ts = cache.tables()
        resident = _np.flatnonzero(k2s >= 0)
        assert len(resident) <= C
        assert all(sk[k2s[key]] == key for key in resident)
        assert all(k2s[sk[s]] == s for s in range(C) if sk[s] >= 0)
        for s, (key, when) in last_use.items():
            if sk[s] == key:
                assert ts[s] == when, (t, s)


def test_run_decisions_closed_forms():
    """The decision stream of a workload: with every key fitting, each key
    misses exactly once (its first use); a resize to the same size changes
    no decision."""
    import numpy as _np
    from oracle.stream import run_decisions
    rng = _np.random.default_rng(12)
    steps, L, T, E, k = 9, 2, 3, 16, 2
    logits = rng.standard_normal((steps, L, T, E)).astype(_np.float32)
    cache, recs = run_decisions(L, E, k, L * E, logits)
    keys = {l * E + int(e) for _, l, idx, _, _ in recs for e in idx.ravel()}
    assert len(recs) == steps * L and cache.n_miss == len(keys) and cache.n_evict == 0
    a, ra = run_decisions(L, E, k, 12, logits)
    b, rb = run_decisions(L, E, k, 12, logits, resize_step=4, resize_slots=12)
    assert (a.n_miss, a.n_hit, a.n_evict) == (b.n_miss, b.n_hit, b.n_evict)
    assert all(_np.array_equal(x[4].miss_expert, y[4].miss_expert) for x, y in zip(ra, rb))
