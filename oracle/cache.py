"""Global expert slot cache with LRU replacement (oracle).

Definition followed ("FreeToken: Efficient Edge-Native MoE Serving with
Bandwidth-Adaptive Execution", design paragraph and ablation paragraph):
the full routed-expert pool lives in host memory; the GPU holds one elastic
expert cache shared by every MoE layer, whose slots are managed by the logical
(layer, expert) id; per layer one kernel does routing dedup, hit
classification and LRU victim selection; replacement is a *global* LRU over
all layers; the cache is rebuilt at a scheduler safe point when the memory
budget changes.

Readings taken where the pages are silent (each is the plainest
deterministic one):

* Events.  Every call of ``event`` is one layer event t = 0, 1, 2, ...
  (steps outer, layers inner).  The key of expert e at layer l is l*E + e.
* Dedup.  U_t is the ascending list of distinct experts among the batch's
  top-k picks at that layer; each is classified and fetched once per event.
* Hit.  e is a hit iff key (l, e) currently occupies a slot.
* Victims.  Candidates are all slots except (a) the slots of this event's
  hits and (b) the slots used by event t-1 ("pin rule": the previous layer's
  FFN may still be reading them while this layer's misses are copied; there is
  no t-1 pin on the first event and on the first event after a resize).
  Candidates are ordered by (last-use event ascending, slot ascending), empty
  slots having last-use -1, and the first |M| are the victims.  The i-th miss
  (ascending expert id) goes to the i-th victim.  Fewer candidates than
  misses is a capacity error.
* Update.  Each victim's old key (if any) is removed, the miss key inserted,
  and every slot of U_t gets last-use = t.
* Miss rate.  Counted per unique expert per layer event: sum|M| / sum|U|.
* Resize (safe point).  Shrinking to C' keeps the min(occupied, C') entries
  that LRU would evict last (drops the first ones in (last-use, slot)
  order); survivors in slots < C' stay, survivors in slots >= C' move, in
  ascending old-slot order, to the lowest free slots < C'.  Last-use values
  are kept.  Growing adds empty slots.
"""
from __future__ import annotations

import dataclasses

import numpy as np


class CapacityError(RuntimeError):
    """Fewer victim candidates than misses (the slot pool is too small)."""


@dataclasses.dataclass
class Event:
    t: int
    layer: int
    unique: np.ndarray        # int32 [n_u] ascending expert ids
    hit: np.ndarray           # uint8 [n_u]
    unique_slot: np.ndarray   # int32 [n_u] slot holding each unique expert after the event
    miss_expert: np.ndarray   # int32 [n_m] ascending
    miss_slot: np.ndarray     # int32 [n_m] victim slot paired with each miss
    evicted_key: np.ndarray   # int32 [n_m] key that occupied the victim (-1 if empty)


class ExpertCacheOracle:
    def __init__(self, num_layers: int, num_experts: int, num_slots: int):
        self.L, self.E, self.C = num_layers, num_experts, num_slots
        self.key_to_slot = np.full(num_layers * num_experts, -1, dtype=np.int64)
        self.slot_key = np.full(num_slots, -1, dtype=np.int64)
        self.slot_ts = np.full(num_slots, -1, dtype=np.int64)
        self.t = 0
        self.prev_slots: set[int] = set()    # slots used by event t-1 (empty: no pin)
        self.n_unique = self.n_hit = self.n_miss = self.n_evict = 0

    # ---- one layer event --------------------------------------------------
    def event(self, layer: int, topk_idx: np.ndarray) -> Event:
        E = self.E
        unique = sorted({int(e) for e in np.asarray(topk_idx).ravel()})
        keys = [layer * E + e for e in unique]
        hit = [self.key_to_slot[k] >= 0 for k in keys]
        misses = [e for e, h in zip(unique, hit) if not h]
        hit_slots = {int(self.key_to_slot[k]) for k, h in zip(keys, hit) if h}

        excluded = np.zeros(self.C, dtype=bool)
        excluded[list(hit_slots)] = True
        excluded[list(self.prev_slots)] = True
        cand = np.flatnonzero(~excluded)
        # order by (last use ascending, slot ascending); lexsort: last key primary
        cand = cand[np.lexsort((cand, self.slot_ts[cand]))]
        if len(cand) < len(misses):
            raise CapacityError(f"event {self.t}: {len(misses)} misses, {len(cand)} candidate slots")
        victims = [int(s) for s in cand[:len(misses)]]

        evicted = []
        for e, s in zip(misses, victims):
            old = int(self.slot_key[s])
            evicted.append(old)
            if old >= 0:
                self.key_to_slot[old] = -1
                self.n_evict += 1
            self.key_to_slot[layer * E + e] = s
            self.slot_key[s] = layer * E + e

        unique_slot = [int(self.key_to_slot[k]) for k in keys]
        for s in unique_slot:
            self.slot_ts[s] = self.t
        ev = Event(self.t, layer, np.array(unique, dtype=np.int32), np.array(hit, dtype=np.uint8),
                   np.array(unique_slot, dtype=np.int32), np.array(misses, dtype=np.int32),
                   np.array(victims, dtype=np.int32), np.array(evicted, dtype=np.int32))
        self.n_unique += len(unique)
        self.n_hit += sum(hit)
        self.n_miss += len(misses)
        self.prev_slots = set(unique_slot)
        self.t += 1
        return ev

    # ---- safe-point resize ------------------------------------------------
    def resize(self, new_slots: int) -> list[tuple[int, int]]:
        """Resize the pool; returns the (old_slot, new_slot) blob moves."""
        occupied = [s for s in range(self.C) if self.slot_key[s] >= 0]
        order = sorted(occupied, key=lambda s: (int(self.slot_ts[s]), s))
        n_drop = max(0, len(occupied) - new_slots)
        dropped, kept = order[:n_drop], set(order[n_drop:])
        for s in dropped:
            self.key_to_slot[self.slot_key[s]] = -1
            self.n_evict += 1
        free = [s for s in range(min(new_slots, self.C)) if s not in kept]
        free += list(range(self.C, new_slots))
        movers = sorted(s for s in kept if s >= new_slots)
        moves = list(zip(movers, free[:len(movers)]))

        new_key = np.full(new_slots, -1, dtype=np.int64)
        new_ts = np.full(new_slots, -1, dtype=np.int64)
        dest = {s: s for s in kept if s < new_slots}
        dest.update(dict(moves))
        for old, new in dest.items():
            new_key[new] = self.slot_key[old]
            new_ts[new] = self.slot_ts[old]
            self.key_to_slot[self.slot_key[old]] = new
        self.slot_key, self.slot_ts, self.C = new_key, new_ts, new_slots
        self.prev_slots = set()
        return moves

    # ---- helpers ----------------------------------------------------------
    def miss_rate(self) -> float:
        return self.n_miss / max(1, self.n_unique)

    def tables(self):
        """(key_to_slot [L*E], slot_key [C], slot_ts [C]) as int32 copies."""
        return (self.key_to_slot.astype(np.int32), self.slot_key.astype(np.int32), self.slot_ts.astype(np.int32))
