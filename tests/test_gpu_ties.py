"""Routing and cache decisions at full width (256 experts, top-8) on
tie-heavy logits, through libft against the oracle.

The logits are multiples of 0.25 (rounded N(0,1)), so most rows hold many
equal values, including equal values among the top 8; each row also gets
three NaN logits (ordered as -inf), one -0.0 and one +0.0 (equal as floats,
so the lower index wins).  This runs the route kernel's 8-logits-per-lane
variant that the 256-expert workloads use, on one CTA (1 and 4 tokens) and on
the multi-CTA path whose last CTA merges the others' bit sets and counts
(64 tokens).  Top-k indices, the unique set, hits, victims, evicted keys and
the slot tables must be bit-exact at every event; gates within 2e-6.  Only
the routing and cache decisions run (no fetch or FFN), so the tables evolve
exactly as the oracle's decision stream.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import routing as orouting
from oracle.cache import ExpertCacheOracle
from synth import workloads as W

pytestmark = pytest.mark.gpu


def tie_logits(seed, steps, L, T, E):
    lg = synth.router_ties(seed, 5, (steps, L, T, E))
    rng = np.random.default_rng(seed)
    for s in range(steps):
        for l in range(L):
            for t in range(T):
                pos = rng.choice(E, 5, replace=False)
                lg[s, l, t, pos[:3]] = np.nan
                lg[s, l, t, pos[3]] = -0.0
                lg[s, l, t, pos[4]] = 0.0
    return lg


@pytest.mark.parametrize("T,C,steps", [(1, 40, 60), (4, 100, 40), (64, 600, 12)], ids=["t1", "t4", "t64-multicta"])
def test_full_width_ties_nan_and_signed_zero(T, C, steps):
    from expert_cache_host_layer_gb300.pipeline import ExpertCache
    from tests.harness import compare_event, make_bank
    L, E, k = 3, 256, 8
    w = W.QWEN35B_DECODE.replace(num_layers=L, hidden=128, inter=128, tokens=T, num_slots=C)
    bank, n_blobs = make_bank(w, 1)
    dev = torch.device("cuda:0")
    cache = ExpertCache(L, E, k, w.hidden, w.inter, w.wdtype, C, T, bank, n_blobs, device=dev)
    ref = ExpertCacheOracle(L, E, C)
    lg = tie_logits(31 + T, steps, L, T, E)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gw = torch.empty((T, k), dtype=torch.float32, device=dev)
    ties_in_topk = 0
    try:
        for s in range(steps):
            for l in range(L):
                cache.route_classify(l, torch.from_numpy(np.ascontiguousarray(lg[s, l])).to(dev), idx, gw)
                ridx, rw = orouting.route(lg[s, l], k)
                ev = ref.event(l, ridx)
                plan = cache.plan(l)
                errs = compare_event(plan, ev, idx.cpu().numpy(), ridx, gw.cpu().numpy(), rw)
                assert not errs, f"step {s} layer {l}: {errs[:3]}"
                sel = np.take_along_axis(lg[s, l], ridx.astype(np.int64), axis=1)
                ties_in_topk += int((np.diff(sel, axis=1) == 0).sum())
            k2s, sk, ts = cache.tables()
            rk, rs, rt = ref.tables()
            assert (k2s == rk).all() and (sk == rs).all() and (ts == rt).all(), f"step {s}"
        assert ties_in_topk > steps * L * T  # ties inside the selected 8 are common, not incidental
        assert ref.n_evict > 0
    finally:
        cache.close()
