"""Cache policies the method is compared with, simulated on the same routing
traces (oracle; test infrastructure, like the rest of this package).

The pages contrast the global (layer, expert) LRU cache with static
placements:
- layer-based offload, which keeps whole layers on the GPU and reads the rest
  from host memory ("FreeToken: az VRAM ile büyük MoE modelleri", the engine
  comparison);
- static expert placement that cannot follow routing which changes from token
  to token ("FreeToken: Efficient Edge-Native MoE Serving ...", motivation
  paragraph);
- keeping a fixed share of experts resident (the --offload-ratio flag of the
  FreeToken MoE inference guide).

Readings:
- Every policy gets the same C slots.
- A miss is a unique (layer, expert) of a layer event that is not resident.
- Static policies are preloaded and never evict; their misses are streamed
  and not kept.
- The static split gives each layer floor(C/L) slots (the first C mod L
  layers one more) and runs an LRU inside each layer.  There is no pin:
  layers do not share slots.
"""
from __future__ import annotations

from collections import OrderedDict

import numpy as np


def unique_events(topk_trace):
    """[(layer, sorted unique experts)] in event order, from top-k indices
    shaped [steps][L][T][k]."""
    steps, L = topk_trace.shape[0], topk_trace.shape[1]
    return [(l, np.unique(topk_trace[s, l])) for s in range(steps) for l in range(L)]


def static_split_lru(events, num_layers: int, num_slots: int):
    """Per-layer LRU caches of floor(C/L) (+1 for the first C mod L layers)
    slots.  Returns (misses, unique)."""
    cap = [num_slots // num_layers + (1 if l < num_slots % num_layers else 0) for l in range(num_layers)]
    caches = [OrderedDict() for _ in range(num_layers)]
    misses = unique = 0
    for l, experts in events:
        c = caches[l]
        for e in experts:
            unique += 1
            if e in c:
                c.move_to_end(e)
                continue
            misses += 1
            if cap[l] == 0:
                continue
            if len(c) >= cap[l]:
                # evict the least recently used expert that this event does not use
                victim = next((k for k in c if k not in set(experts.tolist())), None)
                if victim is None:
                    continue
                del c[victim]
            c[e] = True
    return misses, unique


def static_layers(events, num_layers: int, num_experts: int, num_slots: int):
    """Whole layers resident, the first floor(C/E) of them (layer-based
    offload).  Returns (misses, unique)."""
    resident = num_slots // num_experts
    misses = unique = 0
    for l, experts in events:
        unique += len(experts)
        if l >= resident:
            misses += len(experts)
    return misses, unique


def static_profile(events, num_experts: int, num_slots: int, profile_events: int):
    """The num_slots (layer, expert) keys used most often in the first
    `profile_events` events stay resident (ties: lower key first); measured on
    the events after the profile.  Returns (misses, unique)."""
    counts = {}
    for l, experts in events[:profile_events]:
        for e in experts:
            key = l * num_experts + int(e)
            counts[key] = counts.get(key, 0) + 1
    ranked = sorted(counts.items(), key=lambda kv: (-kv[1], kv[0]))
    resident = {key for key, _ in ranked[:num_slots]}
    misses = unique = 0
    for l, experts in events[profile_events:]:
        for e in experts:
            unique += 1
            misses += (l * num_experts + int(e)) not in resident
    return misses, unique


def previous_step_prefetch_coverage(topk_trace, num_layers: int, num_experts: int, num_slots: int):
    """How many of the global LRU cache's misses a prefetch predicted from the
    previous step's routing could have hidden (the FreeToken MoE inference
    guide, "FreeToken 解决的问题": the engine predicts the experts the next
    token needs and streams them early).

    Reading: the predictor for (step s, layer l) is the unique experts layer l
    used at step s-1; a predicted expert helps only if it is not resident when
    step s reaches layer l (a resident one would hit anyway).  The cache is the
    method's global LRU (ExpertCacheOracle).  Returns (misses, covered,
    predicted_not_resident): the misses, the misses that were predicted, and
    the predicted experts that were not resident (the prefetch traffic it would
    add, useful or not)."""
    from .cache import ExpertCacheOracle
    steps = topk_trace.shape[0]
    cache = ExpertCacheOracle(num_layers, num_experts, num_slots)
    prev = [None] * num_layers
    misses = covered = wasted_or_useful = 0
    for s in range(steps):
        for l in range(num_layers):
            pred = prev[l]
            if pred is not None:
                not_res = {int(e) for e in pred if cache.key_to_slot[l * num_experts + int(e)] < 0}
            else:
                not_res = set()
            ev = cache.event(l, topk_trace[s, l])
            m = {int(e) for e in ev.miss_expert}
            if s > 0:  # the first step has no predictor
                misses += len(m)
                covered += len(m & not_res)
                wasted_or_useful += len(not_res)
            prev[l] = np.unique(topk_trace[s, l])
    return misses, covered, wasted_or_useful


def frequency_prefetch_coverage(topk_trace, num_layers: int, num_experts: int, num_slots: int, per_layer: int,
                                warm_steps: int = 0):
    """How many of the global LRU cache's misses a prefetch of each layer's
    most often used experts could have hidden, and how much link traffic it
    would add (the same page as previous_step_prefetch_coverage: predict the
    next experts and stream them early; here the predictor is the routing
    history instead of the last step).

    Reading: before step s reaches layer l, the predictor names the
    `per_layer` experts of layer l with the most uses in steps < s (ties: lower
    expert index) among those not resident at that moment; a miss of that
    event is covered if its expert was named.  Counted from step
    `warm_steps` on.  Returns (misses, covered, prefetched)."""
    from .cache import ExpertCacheOracle
    steps = topk_trace.shape[0]
    cache = ExpertCacheOracle(num_layers, num_experts, num_slots)
    uses = np.zeros((num_layers, num_experts), dtype=np.int64)
    misses = covered = prefetched = 0
    for s in range(steps):
        for l in range(num_layers):
            order = sorted(range(num_experts), key=lambda e: (-uses[l, e], e))
            named = [e for e in order if cache.key_to_slot[l * num_experts + e] < 0][:per_layer]
            ev = cache.event(l, topk_trace[s, l])
            if s >= warm_steps:
                m = {int(e) for e in ev.miss_expert}
                misses += len(m)
                covered += len(m & set(named))
                prefetched += len(named)
            for e in np.unique(topk_trace[s, l]):
                uses[l, int(e)] += 1
    return misses, covered, prefetched
