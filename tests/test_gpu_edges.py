"""GPU edge cases and error paths of the C ABI (no case faults the GPU: every
error is caught on the host before a launch, or is a capacity condition the
kernel reports through its status word)."""
import numpy as np
import pytest
import torch

import synth
from oracle import routing as orouting
from oracle.cache import ExpertCacheOracle
from synth import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import expert_cache_host_layer_gb300 as ft
    from expert_cache_host_layer_gb300.pipeline import ExpertCache
    from tests.harness import make_bank


def small_cache(E=16, k=2, L=2, C=12, T=1, H=256, I=128, wdtype=synth.W_F32, mode=1):
    w = W.TINY.replace(num_experts=E, top_k=k, num_layers=L, num_slots=C, tokens=T, hidden=H, inter=I, wdtype=wdtype)
    bank, n = make_bank(w, min(w.blobs, 64))
    return w, ExpertCache(L, E, k, H, I, wdtype, C, T, bank, n, fetch_mode=mode)


def test_capacity_bound_rejected_at_create():
    w = W.TINY
    bank, n = make_bank(w, 4)
    with pytest.raises(ft.FtError) as e:
        ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, 3, 1, bank, 4)
    assert e.value.status == ft.FT_ERR_CAPACITY


def test_call_order_errors():
    w, c = small_cache()
    dev = torch.device("cuda:0")
    x = torch.zeros((1, w.hidden), device=dev)
    y = torch.zeros_like(x)
    with pytest.raises(ft.FtError) as e:
        c.moe_forward(0, x, y)                       # nothing classified
    assert e.value.status == ft.FT_ERR_STATE
    with pytest.raises(ft.FtError) as e:
        c.fetch_misses(1)
    assert e.value.status == ft.FT_ERR_STATE
    lg = torch.randn((1, w.num_experts), device=dev)
    c.route_classify(0, lg)
    with pytest.raises(ft.FtError) as e:
        c.moe_forward(0, x, y)                       # classified, not fetched
    assert e.value.status == ft.FT_ERR_STATE
    c.fetch_misses(0)
    with pytest.raises(ft.FtError) as e:
        c.route_classify(0, lg)                      # fetched plan not yet consumed
    assert e.value.status == ft.FT_ERR_STATE
    with pytest.raises(ft.FtError) as e:
        c.moe_forward(0, torch.zeros((2, w.hidden), device=dev), y)  # T differs from the plan
    assert e.value.status == ft.FT_ERR_INVALID_ARG
    c.moe_forward(0, x, y)
    with pytest.raises(ft.FtError) as e:
        c.route_classify(5, lg)
    assert e.value.status == ft.FT_ERR_INVALID_ARG
    c.synchronize()
    c.close()


def test_only_one_layer_may_run_ahead():
    w, c = small_cache(L=3)
    dev = torch.device("cuda:0")
    lg = torch.randn((1, w.num_experts), device=dev)
    c.route_classify(0, lg); c.fetch_misses(0)
    c.route_classify(1, lg); c.fetch_misses(1)
    with pytest.raises(ft.FtError) as e:   # event 0 still unconsumed two events later
        c.route_classify(2, lg)
    assert e.value.status == ft.FT_ERR_STATE
    x = torch.zeros((1, w.hidden), device=dev)
    c.moe_forward(0, x, torch.empty_like(x))
    c.route_classify(2, lg)
    c.close()


def test_empty_batch_and_all_experts_selected():
    w, c = small_cache(E=16, k=16, C=32)
    dev = torch.device("cuda:0")
    ref = ExpertCacheOracle(w.num_layers, 16, 32)
    lg = synth.normal(synth.key(3), 5 * 16).reshape(5, 1, 16)
    for i in range(5):
        layer = i % 2
        if i == 2:  # empty batch
            c.route_classify(layer, torch.empty((0, 16), device=dev))
            ev = ref.event(layer, np.zeros((0, 16), dtype=np.int32))
        else:
            c.route_classify(layer, torch.from_numpy(lg[i]).to(dev))
            ev = ref.event(layer, orouting.topk(lg[i], 16))
        p = c.plan(layer)
        assert p["unique"].tolist() == ev.unique.tolist()
        assert p["miss_slot"].tolist() == ev.miss_slot.tolist()
        assert p["evicted_key"].tolist() == ev.evicted_key.tolist()
        c.fetch_misses(layer)
        x = torch.zeros((0 if i == 2 else 1, w.hidden), device=dev)
        c.moe_forward(layer, x, torch.empty_like(x))
    k2s, sk, ts = c.tables()
    rk, rs, rt = ref.tables()
    assert (k2s == rk).all() and (sk == rs).all() and (ts == rt).all()
    c.close()


def test_nan_logits_ordered_as_minus_inf():
    w, c = small_cache()
    dev = torch.device("cuda:0")
    row = np.array([[np.nan, 0.5, np.nan, -0.0, 0.0, 3.0] + [-np.inf] * 10], dtype=np.float32)
    idx = torch.empty((1, 2), dtype=torch.int32, device=dev)
    c.route_classify(0, torch.from_numpy(row).to(dev), idx)  # noqa
    torch.cuda.synchronize()
    assert idx.cpu().numpy().tolist() == orouting.topk(row, 2).tolist() == [[5, 1]]
    c.close()


def test_resize_grow_and_to_new_pool():
    w = W.TINY
    bank, n = make_bank(w)
    c = ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, 12, 1, bank, n)
    ref = ExpertCacheOracle(w.num_layers, w.num_experts, 12)
    dev = torch.device("cuda:0")
    lg = W.router_logits(w.replace(steps=30))
    x = torch.zeros((1, w.hidden), device=dev)
    y = torch.empty_like(x)
    for s in range(30):
        if s == 10:
            c.resize(20)                    # grow into a new pool
            ref.resize(20)
        if s == 20:
            newpool = torch.empty(6 * c.eb, dtype=torch.uint8, device=dev)
            c.resize(6, newpool)            # shrink into another pool: all survivors copied
            ref.resize(6)
        for l in range(w.num_layers):
            c.route_classify(l, torch.from_numpy(lg[s, l]).to(dev))
            ref.event(l, orouting.topk(lg[s, l], w.top_k))
            c.fetch_misses(l)
            c.moe_forward(l, x, y)
        k2s, sk, ts = c.tables()
        rk, rs, rt = ref.tables()
        assert (k2s == rk).all() and (sk == rs).all() and (ts == rt).all(), f"step {s}"
    # every occupied slot holds its key's blob
    for slot in range(6):
        key = int(sk[slot])
        if key >= 0:
            got = c.pool[slot * c.eb:(slot + 1) * c.eb].cpu().numpy()
            b = key % n
            assert np.array_equal(got, bank.numpy()[b * c.eb:(b + 1) * c.eb])
    c.close()


def test_copy_thread_never_served_times_out_and_next_cache_works():
    """Copy-engine mode with the library's copy thread paused: the layer's FFN
    kernel waits for copies that never come, gives up after its bounded wait
    (about one second), records FT_ERR_TIMEOUT and finishes; ft_synchronize
    reports it once the thread resumes.  The GPU stays usable: a new cache
    then runs a short decode in parity with the oracle."""
    import time
    w = W.TINY
    bank, n = make_bank(w)
    dev = torch.device("cuda:0")
    c = ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, w.num_slots, 1, bank, n,
                    fetch_mode=ft.FT_FETCH_COPY_ENGINE, device=dev)
    try:
        ft.ft_debug_pause_copies(c.handle, True)
        lg = torch.from_numpy(W.router_logits(w.replace(steps=1))[0, 0]).to(dev)
        x = torch.zeros((1, w.hidden), device=dev)
        y = torch.empty_like(x)
        c.route_classify(0, lg)
        c.fetch_misses(0)                   # a cold cache: every pick misses
        c.moe_forward(0, x, y)
        t0 = time.monotonic()
        while time.monotonic() - t0 < 5.0 and torch.cuda.current_stream(dev).query() is False:
            time.sleep(0.05)                # the FFN's own bounded wait ends it
        assert torch.cuda.current_stream(dev).query(), "FFN kernel still running 5 s after its 1 s wait limit"
        ft.ft_debug_pause_copies(c.handle, False)
        with pytest.raises(ft.FtError) as e:
            c.synchronize()
        assert e.value.status == ft.FT_ERR_TIMEOUT
    finally:
        c.close()
    from tests.harness import run_parity
    rep = run_parity(w, steps=4, fetch_mode=0)
    assert rep["events"] == 8


def test_budget_shrink_and_regrow_mid_stream_matches_oracle():
    """A 35B-shaped cache sized from a byte budget, shrunk to a smaller budget
    after 10 steps (into a new, smaller pool: the memory goes back) and grown
    to a larger one after 20, at safe points; decisions and tables against the
    oracle given the same slot counts, fetched slots against the bank."""
    w = W.QWEN35B_DECODE.replace(num_layers=6)
    bank, n = make_bank(w, 256)
    dev = torch.device("cuda:0")
    eb = w.expert_bytes
    budgets = [400 * eb, 130 * eb, 700 * eb]
    c = ExpertCache.from_budget(budgets[0], w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, 1,
                                bank, n, device=dev)
    sizes = [c.num_slots]
    assert c.device_bytes() <= budgets[0] < c.device_bytes() + eb
    ref = ExpertCacheOracle(w.num_layers, w.num_experts, c.num_slots)
    lg = W.router_logits(w.replace(steps=30))
    x = torch.zeros((1, w.hidden), dtype=torch.bfloat16, device=dev)
    y = torch.empty((1, w.hidden), dtype=torch.float32, device=dev)
    try:
        for s in range(30):
            if s in (10, 20):
                slots = c.resize_to_budget(budgets[1 if s == 10 else 2])
                ref.resize(slots)
                sizes.append(slots)
            for l in range(w.num_layers):
                c.route_classify(l, torch.from_numpy(lg[s, l]).to(dev))
                ev = ref.event(l, orouting.topk(lg[s, l], w.top_k))
                p = c.plan(l)
                assert p["miss_slot"].tolist() == ev.miss_slot.tolist(), (s, l)
                assert p["evicted_key"].tolist() == ev.evicted_key.tolist(), (s, l)
                c.fetch_misses(l)
                c.moe_forward(l, x, y)
            k2s, sk, ts = c.tables()
            rk, rs, rt = ref.tables()
            assert (k2s == rk).all() and (sk == rs).all() and (ts == rt).all(), f"step {s}"
        assert sizes[1] < sizes[0] < sizes[2]
        c.synchronize()
        for slot in range(0, c.num_slots, 97):   # every fetched slot holds its key's blob
            key = int(sk[slot])
            if key >= 0:
                got = c.pool[slot * eb:(slot + 1) * eb].cpu().numpy()
                b = key % n
                assert np.array_equal(got, bank.numpy()[b * eb:(b + 1) * eb]), slot
    finally:
        c.close()
