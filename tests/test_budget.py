"""Budget-driven cache sizing (ft_slots_for_budget, ft_cache_overhead_bytes):
host arithmetic only, so these run without a GPU.

The pages size the cache automatically from the free device memory ("FreeToken
vs vLLM on one RTX 3090", Runtime configurations) and rebuild it when the
budget changes ("FreeToken: Efficient Edge-Native MoE Serving ...", design
paragraph).  Checked here: the returned slot count is the largest whose pool
plus the library's own allocations fit, the overhead grows with the slot
count, and a budget below the capacity bound is refused.
"""
import pytest

import expert_cache_host_layer_gb300 as ft


def cfg(L=40, E=256, k=8, H=2048, I=512, wd=ft.FT_W_BF16, T=1, mode=ft.FT_FETCH_SM_PULL):
    return ft.make_config(L, E, k, H, I, wd, 0, 0, 1, T, mode)


@pytest.mark.parametrize("c", [cfg(), cfg(T=8), cfg(T=16384), cfg(L=24, H=4096, I=2048, wd=ft.FT_W_FP8E4M3_B128),
                               cfg(L=2, E=16, k=2, H=256, I=128, wd=ft.FT_W_F32, mode=ft.FT_FETCH_COPY_ENGINE)])
def test_slots_for_budget_is_the_largest_that_fits(c):
    eb = ft.ft_expert_bytes(c.hidden, c.inter, c.wdtype)
    for budget in (64 * eb + (1 << 24), 1000 * eb + 12345, 3072 * eb + (7 << 20), 10 ** 11):
        try:
            n = ft.ft_slots_for_budget(c, budget)
        except ft.FtError as e:
            assert e.status == ft.FT_ERR_CAPACITY
            continue
        assert n * eb + ft.ft_cache_overhead_bytes(c, n) <= budget
        assert (n + 1) * eb + ft.ft_cache_overhead_bytes(c, n + 1) > budget


def test_overhead_grows_with_slots_and_counts_the_prefill_buffers():
    c = cfg()
    prev = 0
    for n in (16, 100, 1000, 3072, 20000):
        o = ft.ft_cache_overhead_bytes(c, n)
        assert o >= prev
        prev = o
    # a 16,384-token chunk needs the grouped x rows, h and the per-row outputs (all 16-bit) for
    # 131,072 rows: far more than decode
    rows = 131072
    assert ft.ft_cache_overhead_bytes(cfg(T=16384), 3072) > \
        ft.ft_cache_overhead_bytes(c, 3072) + rows * (2048 * 2 + 512 * 2 + 2048 * 2)
    assert ft.ft_cache_overhead_bytes(c, 0) == 0


def test_budget_below_the_capacity_bound_is_refused():
    c = cfg(T=8)                     # bound = 2 * min(64, 256) = 128 slots
    eb = ft.ft_expert_bytes(2048, 512, ft.FT_W_BF16)
    with pytest.raises(ft.FtError) as e:
        ft.ft_slots_for_budget(c, 127 * eb)
    assert e.value.status == ft.FT_ERR_CAPACITY
    assert ft.ft_slots_for_budget(c, 200 * eb) >= 128
