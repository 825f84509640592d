"""ft_moe_decode_ffn_static: the decode FFN entry point that allocates nothing.

It exists for callers that may not allocate device memory (a memory planner
that owns all of it, or a serving loop that cannot afford a cudaMalloc or
cudaFree stall); its working memory is a static device array inside libft.
This test calls it through the C ABI and checks its output against
ft_moe_forward (the cache path) on the same weights, routing and inputs, on
two calls in a row (the second call reuses the array the first one left
behind).  It also checks that sizes beyond the array are rejected before any
GPU work.  Collected last so a stop-at-first-failure run has already run the
other tests; it needs no state from them.
"""
import numpy as np
import pytest
import torch

import synth
from synth import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import expert_cache_host_layer_gb300 as ft
    from expert_cache_host_layer_gb300.pipeline import ExpertCache
    from tests.harness import TOL, make_bank, to_act


@pytest.mark.parametrize("w", [W.TINY, W.QWEN35B_DECODE_B4], ids=["tiny-fp32", "qwen35b-b4-bf16"])
def test_static_ffn_matches_cache_forward_two_calls(w):
    dev = torch.device("cuda:0")
    bank, n_blobs = make_bank(w, min(w.blobs, 256))
    cache = ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, w.num_slots, w.tokens,
                        bank, n_blobs, device=dev)
    logits = W.router_logits(w.replace(steps=3))
    T, k, E = w.tokens, w.top_k, w.num_experts
    try:
        calls = 0
        for s in range(3):
            for l in range(2):                       # two consecutive layer events per step
                lg = torch.from_numpy(np.ascontiguousarray(logits[s, l])).to(dev)
                idx = torch.empty((T, k), dtype=torch.int32, device=dev)
                gw = torch.empty((T, k), dtype=torch.float32, device=dev)
                x = to_act(W.hidden_states(w, s, l), w, dev)
                y_ref = torch.empty((T, w.hidden), dtype=torch.float32, device=dev)
                cache.route_classify(l, lg, idx, gw)
                cache.fetch_misses(l)
                cache.moe_forward(l, x, y_ref)
                cache.synchronize()
                k2s, _, _ = cache.tables()
                expert_slot = torch.from_numpy(np.ascontiguousarray(k2s[l * E:(l + 1) * E])).to(dev)
                y = torch.full((T, w.hidden), float("nan"), dtype=torch.float32, device=dev)
                ft.ft_moe_decode_ffn_static(w.hidden, w.inter, w.wdtype, E, k, cache.pool.data_ptr(),
                                            cache.num_slots, expert_slot.data_ptr(), idx.data_ptr(),
                                            gw.data_ptr(), x.data_ptr(), T, y.data_ptr(),
                                            torch.cuda.current_stream(dev).cuda_stream)
                torch.cuda.synchronize(dev)
                yr = y_ref.float().cpu().numpy().astype(np.float64)
                yg = y.float().cpu().numpy().astype(np.float64)
                rms = np.sqrt(np.mean(yr ** 2))
                assert np.isfinite(yg).all()
                assert np.abs(yg - yr).max() <= TOL[w.wdtype] * rms, (s, l)
                calls += 1
        assert calls == 6
    finally:
        cache.close()


def test_static_ffn_rejects_sizes_beyond_its_array():
    p = 1 << 20  # never dereferenced: the size checks come first
    with pytest.raises(ft.FtError) as e:   # T beyond the decode limit
        ft.ft_moe_decode_ffn_static(2048, 512, ft.FT_W_BF16, 256, 8, p, 10, p, p, p, p, 9, p)
    assert e.value.status == ft.FT_ERR_INVALID_ARG and "T=9" in str(e.value)
    with pytest.raises(ft.FtError) as e:   # 8 * 32 rows * 2048 * 4 B of intermediate > 1 MiB array
        ft.ft_moe_decode_ffn_static(4096, 2048, ft.FT_W_FP8E4M3_B128, 256, 32, p, 10, p, p, p, p, 8, p)
    assert e.value.status == ft.FT_ERR_INVALID_ARG and "static scratch" in str(e.value)
