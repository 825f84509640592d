"""The decision stream of a whole workload (oracle).

Layer events run in the order steps outer, layers inner, which is also the
order the library assigns event numbers.  Before step `resize_step` the cache
is resized at a safe point ("FreeToken: Efficient Edge-Native MoE Serving
...", design paragraph: cache rebuilt at scheduler safe points without
restarting the engine).
"""
from __future__ import annotations

import numpy as np

from . import routing
from .cache import ExpertCacheOracle


def run_decisions(num_layers: int, num_experts: int, top_k: int, num_slots: int, logits: np.ndarray,
                  resize_step: int = -1, resize_slots: int = 0, keep_events: bool = True):
    """Replay routing + cache decisions for logits [steps][L][T][E].

    Returns (cache, records) where records[i] = (step, layer, topk_idx, gates,
    Event) for each event i (records is empty when keep_events is False), and
    the moves of the resize (if any) are stored in cache.resize_moves.
    """
    cache = ExpertCacheOracle(num_layers, num_experts, num_slots)
    cache.resize_moves = []
    records = []
    steps = logits.shape[0]
    for s in range(steps):
        if s == resize_step:
            cache.resize_moves = cache.resize(resize_slots)
        for l in range(num_layers):
            idx, w = routing.route(logits[s, l], top_k)
            ev = cache.event(l, idx)
            if keep_events:
                records.append((s, l, idx, w, ev))
    return cache, records
