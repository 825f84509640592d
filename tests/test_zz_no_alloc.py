"""ft_moe_decode_ffn_static: the decode FFN entry point that allocates nothing.

It exists for callers that may not allocate device memory (a memory planner
that owns all of it, or a serving loop that cannot afford a cudaMalloc or
cudaFree stall); its working memory is a static device array inside libft.
These tests call it through the C ABI and check its output on two calls in a
row (the second call reuses the array the first one left behind):

* against ft_moe_forward (the cache path) on the same weights, routing and
  inputs, within the FFN tolerance;
* against the CPU oracle's FFN, element by element, on fp32, bf16 and fp8
  block-scaled experts;
* with picks the entry point must skip (expert id -1 or past E, an expert
  whose slot is -1): the oracle's FFN with those picks dropped.

It also checks that sizes beyond the array, and a hidden size the kernels
cannot split, are rejected before any GPU work, and that the status word
reads clean after the calls.  Collected last so a stop-at-first-failure run
has already run the other tests; it needs no state from them.
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
    from tests.harness import TOL, bank_blob, ffn_error, make_bank, to_act
    from oracle import ffn as offn

# an fp8 block-scaled shape whose intermediate fits the static array: 4 tokens x 4 picks x 256
FP8_SMALL = W.TINY.replace(name="fp8-small-b4", num_experts=16, top_k=4, hidden=512, inter=256,
                           wdtype=synth.W_FP8, tokens=4, num_slots=32)


def static_call(w, cache_pool, num_slots, expert_slot, idx, gw, x, y, dev):
    ft.ft_moe_decode_ffn_static(w.hidden, w.inter, w.wdtype, w.num_experts, w.top_k, cache_pool, num_slots,
                                expert_slot.data_ptr(), idx.data_ptr(), gw.data_ptr(), x.data_ptr(), w.tokens,
                                y.data_ptr(), torch.cuda.current_stream(dev).cuda_stream)


def oracle_y(w, bank, n_blobs, layer, x_h, idx_h, gw_h, valid):
    """The oracle FFN over the valid picks only (the others contribute nothing)."""
    T, k = idx_h.shape
    y = np.zeros((T, w.hidden))
    weights = {}
    for t in range(T):
        for j in range(k):
            if not valid[t, j]:
                continue
            e = int(idx_h[t, j])
            if e not in weights:
                weights[e] = offn.dequant_blob(bank_blob(bank, w, n_blobs, layer, e), w.hidden, w.inter, w.wdtype)
            y[t] += gw_h[t, j] * offn.expert_ffn(x_h[t:t + 1].astype(np.float64), *weights[e])[0]
    return y


@pytest.mark.parametrize("w", [W.TINY, W.QWEN35B_DECODE_B4, FP8_SMALL], ids=["tiny-fp32", "qwen35b-b4-bf16",
                                                                          "fp8-small-b4"])
def test_static_ffn_matches_cache_forward_and_oracle_two_calls(w):
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
                x_h = W.hidden_states(w, s, l)
                x = to_act(x_h, w, dev)
                y_ref = torch.empty((T, w.hidden), dtype=torch.float32, device=dev)
                cache.route_classify(l, lg, idx, gw)
                cache.fetch_misses(l)
                cache.moe_forward(l, x, y_ref)
                cache.synchronize()
                k2s, _, _ = cache.tables()
                expert_slot = torch.from_numpy(np.ascontiguousarray(k2s[l * E:(l + 1) * E])).to(dev)
                y = torch.full((T, w.hidden), float("nan"), dtype=torch.float32, device=dev)
                static_call(w, cache.pool.data_ptr(), cache.num_slots, expert_slot, idx, gw, x, y, dev)
                torch.cuda.synchronize(dev)
                yr = y_ref.float().cpu().numpy().astype(np.float64)
                yg = y.float().cpu().numpy().astype(np.float64)
                rms = np.sqrt(np.mean(yr ** 2))
                assert np.isfinite(yg).all()
                assert np.abs(yg - yr).max() <= TOL[w.wdtype] * rms, (s, l)
                # and against the oracle (x as the kernels see it: bf16-rounded for bf16/fp8 experts)
                x_seen = x.float().cpu().numpy().astype(np.float64)
                yo = oracle_y(w, bank, n_blobs, l, x_seen, idx.cpu().numpy(), gw.cpu().numpy().astype(np.float64),
                              np.ones((T, k), dtype=bool))
                mx, _ = ffn_error(yg, yo)
                assert mx <= TOL[w.wdtype], (s, l, mx)
                calls += 1
        assert calls == 6
        ft.ft_moe_decode_ffn_static_status(torch.cuda.current_stream(dev).cuda_stream)
    finally:
        cache.close()


@pytest.mark.parametrize("w", [W.TINY, FP8_SMALL], ids=["tiny-fp32", "fp8-small-b4"])
def test_static_ffn_skips_invalid_picks(w):
    """Picks with an expert id of -1 or past E, and an expert whose slot is -1,
    contribute nothing; two calls in a row on the same array."""
    dev = torch.device("cuda:0")
    bank, n_blobs = make_bank(w, min(w.blobs, 256))
    T, k, E = w.tokens, w.top_k, w.num_experts
    layer = 1
    # a hand-made pool: expert e of `layer` in slot (E - 1 - e); expert 3 has no slot
    eb = w.expert_bytes
    pool_h = np.zeros(E * eb, dtype=np.uint8)
    slot_of = np.array([E - 1 - e for e in range(E)], dtype=np.int32)
    slot_of[3] = -1
    for e in range(E):
        if slot_of[e] >= 0:
            pool_h[slot_of[e] * eb:(slot_of[e] + 1) * eb] = bank_blob(bank, w, n_blobs, layer, e)
    pool = torch.from_numpy(pool_h).to(dev)
    expert_slot = torch.from_numpy(slot_of).to(dev)
    rng = np.random.default_rng(17)
    for call in range(2):
        idx_h = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        idx_h[0, 0] = -1
        idx_h[min(1, T - 1), k - 1] = E + 1
        idx_h[T - 1, 0] = 3                           # an expert with no slot
        gw_h = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
        x_h = W.hidden_states(w, 5 + call, layer)
        x = to_act(x_h, w, dev)
        idx = torch.from_numpy(idx_h).to(dev)
        gw = torch.from_numpy(gw_h).to(dev)
        y = torch.full((T, w.hidden), float("nan"), dtype=torch.float32, device=dev)
        static_call(w, pool.data_ptr(), E, expert_slot, idx, gw, x, y, dev)
        torch.cuda.synchronize(dev)
        valid = (idx_h >= 0) & (idx_h < E)
        valid &= np.where(valid, slot_of[np.clip(idx_h, 0, E - 1)] >= 0, False)
        assert not valid.all()
        x_seen = x.float().cpu().numpy().astype(np.float64)
        yo = oracle_y(w, bank, n_blobs, layer, x_seen, idx_h, gw_h.astype(np.float64), valid)
        yg = y.cpu().numpy().astype(np.float64)
        assert np.isfinite(yg).all()
        mx, _ = ffn_error(yg, yo)
        assert mx <= TOL[w.wdtype], (call, mx)
    ft.ft_moe_decode_ffn_static_status(torch.cuda.current_stream(dev).cuda_stream)


def test_static_ffn_rejects_sizes_beyond_its_array():
    p = 1 << 20  # never dereferenced: the size checks come first
    with pytest.raises(ft.FtError) as e:   # T beyond the decode limit
        ft.ft_moe_decode_ffn_static(2048, 512, ft.FT_W_BF16, 256, 8, p, 10, p, p, p, p, 9, p)
    assert e.value.status == ft.FT_ERR_INVALID_ARG and "T=9" in str(e.value)
    with pytest.raises(ft.FtError) as e:   # 8 * 32 rows * 2048 * 4 B of intermediate > 1 MiB array
        ft.ft_moe_decode_ffn_static(4096, 2048, ft.FT_W_FP8E4M3_B128, 256, 32, p, 10, p, p, p, p, 8, p)
    assert e.value.status == ft.FT_ERR_INVALID_ARG and "static scratch" in str(e.value)
    with pytest.raises(ft.FtError) as e:   # fp32 hidden 260: a multiple of 4, not of 8
        ft.ft_moe_decode_ffn_static(260, 128, ft.FT_W_F32, 16, 2, p, 10, p, p, p, p, 1, p)
    assert e.value.status == ft.FT_ERR_INVALID_ARG and "multiple of 8" in str(e.value)
