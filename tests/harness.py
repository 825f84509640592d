"""Side-by-side runner for the GPU parity tests: the CUDA path through the C
ABI on one side, the CPU oracle on the other, on the same seeded inputs.

Nothing here feeds a GPU result into the oracle: the oracle sees only the
generated logits, hidden states and host-bank bytes.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import synth
from oracle import ffn as offn
from oracle import routing as orouting
from oracle.cache import ExpertCacheOracle
from synth import workloads as W

TOL = {synth.W_F32: 1e-4, synth.W_BF16: 2e-2, synth.W_FP8: 2e-2}


def make_bank(w: W.Workload, blobs: int | None = None) -> tuple[torch.Tensor, int]:
    """Pinned host bank of `blobs` generated expert blobs (aliased when < L*E)."""
    from expert_cache_host_layer_gb300.pipeline import pinned_bank
    n = blobs or w.blobs
    bank = pinned_bank(n * w.expert_bytes)
    synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, np.arange(n), out_ptr=bank.data_ptr())
    return bank, n


def bank_blob(bank: torch.Tensor, w: W.Workload, n_blobs: int, layer: int, expert: int) -> np.ndarray:
    b = (layer * w.num_experts + expert) % n_blobs
    eb = w.expert_bytes
    return bank.numpy()[b * eb:(b + 1) * eb]


def shift_fp8_scales(blobs: np.ndarray, w: W.Workload, n_blobs: int, shifts: tuple[int, int, int]) -> None:
    """Multiply every bf16 block scale of Wg, Wu and Wd in `n_blobs` fp8 blobs
    (uint8 array, runtime layout) by 2**shifts[0], 2**shifts[1], 2**shifts[2],
    in place: an exact change of each scale's exponent field.  Both the GPU
    path and the oracle then read the same, still valid, blobs."""
    assert w.wdtype == synth.W_FP8
    H, I, eb = w.hidden, w.inter, w.expert_bytes
    g = (H // 128) * (I // 128)
    for b in range(n_blobs):
        off = b * eb + 3 * H * I
        sc = blobs[off:off + 6 * g].view(np.uint16)
        for m, sh in enumerate(shifts):
            part = sc[m * g:(m + 1) * g]
            e = (part.astype(np.int32) >> 7) & 0xFF
            assert np.all((e == 0) | ((e + sh > 0) & (e + sh < 255))), "scale exponent out of range"
            part[:] = np.where(e == 0, part, part.astype(np.int32) + (sh << 7)).astype(np.uint16)


def to_act(x: np.ndarray, w: W.Workload, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device=device, dtype=torch.float32 if w.wdtype == synth.W_F32 else torch.bfloat16)


@dataclasses.dataclass
class Mismatch:
    what: str
    event: int
    detail: str


def compare_event(plan, ev, gpu_idx, ref_idx, gpu_w, ref_w):
    errs = []
    if not np.array_equal(gpu_idx, ref_idx):
        errs.append(("topk_idx", f"{gpu_idx.tolist()} != {ref_idx.tolist()}"))
    if gpu_w is not None and not np.allclose(gpu_w, ref_w, rtol=0, atol=2e-6):
        errs.append(("topk_w", f"max diff {np.abs(gpu_w - ref_w).max()}"))
    for name, g, r in (("event", plan["event"], ev.t), ("unique", plan["unique"], ev.unique),
                       ("hit", plan["hit"], ev.hit), ("unique_slot", plan["unique_slot"], ev.unique_slot),
                       ("miss_expert", plan["miss_expert"], ev.miss_expert),
                       ("miss_slot", plan["miss_slot"], ev.miss_slot),
                       ("evicted_key", plan["evicted_key"], ev.evicted_key)):
        if not np.array_equal(np.asarray(g), np.asarray(r)):
            errs.append((name, f"gpu {np.asarray(g).tolist()} vs oracle {np.asarray(r).tolist()}"))
    return errs


def ffn_error(y_gpu: np.ndarray, y_ref: np.ndarray) -> tuple[float, float]:
    """(max |diff| / RMS(ref), RMS(diff) / RMS(ref))."""
    rms = float(np.sqrt(np.mean(y_ref ** 2))) or 1.0
    d = y_gpu.astype(np.float64) - y_ref
    return float(np.abs(d).max() / rms), float(np.sqrt(np.mean(d ** 2)) / rms)


def oracle_ffn(w: W.Workload, bank, n_blobs, layer, x, idx, gates):
    cache = {}

    def weights_of(e):
        if e not in cache:
            cache[e] = offn.dequant_blob(bank_blob(bank, w, n_blobs, layer, e), w.hidden, w.inter, w.wdtype)
        return cache[e]

    return offn.moe_ffn(x.astype(np.float64), idx, gates, weights_of)


def run_parity(w: W.Workload, steps: int | None = None, fetch_mode: int = 1, double_buffer: bool = True,
               bank_blobs: int | None = None, check_tables_every: int = 1, ffn_every: int = 1,
               check_slots: bool = True, copy_streams: int = 1, logits=None, device="cuda:0",
               ffn_tokens=None, ffn_workers: int = 0, fp8_scale_shifts=None):
    """Run `steps` steps of workload w through libft and the oracle.

    ffn_tokens: compare the FFN output on these token rows only; a callable
    ffn_tokens(layer, topk_idx) returns the rows for that layer event (None:
    every row).  Decisions are always compared in full.
    fp8_scale_shifts: (Wg, Wu, Wd) powers of two applied to every block scale
    of the bank before the run (shift_fp8_scales).
    ffn_workers: check the FFN outputs in that many spawned host processes
    (tests/oracle_worker.py) while the GPU run goes on; 0 checks inline.  Returns a report dict; raises AssertionError on the
    first mismatch.
    """
    from expert_cache_host_layer_gb300.pipeline import ExpertCache
    steps = steps or w.steps
    dev = torch.device(device)
    bank, n_blobs = make_bank(w, bank_blobs)
    if fp8_scale_shifts is not None:
        shift_fp8_scales(bank.numpy(), w, n_blobs, fp8_scale_shifts)
    if logits is None:
        logits = W.router_logits(w.replace(steps=steps))
    cache = ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, w.num_slots,
                        max(w.tokens, 1), bank, n_blobs, fetch_mode=fetch_mode, copy_streams=copy_streams,
                        device=device)
    ref = ExpertCacheOracle(w.num_layers, w.num_experts, w.num_slots)
    L, T, k = w.num_layers, w.tokens, w.top_k
    idx_d = [torch.empty((T, k), dtype=torch.int32, device=dev) for _ in range(L)]
    wt_d = [torch.empty((T, k), dtype=torch.float32, device=dev) for _ in range(L)]
    ys = [torch.empty((T, w.hidden), dtype=cache.out_dtype, device=dev) for _ in range(L)]
    report = {"events": 0, "ffn_checked": 0, "max_err": 0.0, "max_rms_err": 0.0, "slots_checked": 0}
    ev_counter = [0]
    pool, pending = None, []
    if ffn_workers:
        import concurrent.futures
        import multiprocessing

        from tests import oracle_worker
        pool = concurrent.futures.ProcessPoolExecutor(ffn_workers, mp_context=multiprocessing.get_context("spawn"))

    def check_ffn(t, mx, rm):
        report["max_err"] = max(report["max_err"], mx)
        report["max_rms_err"] = max(report["max_rms_err"], rm)
        report["ffn_checked"] += 1
        assert mx <= TOL[w.wdtype], f"event {t}: FFN max err {mx:.3e} x RMS > {TOL[w.wdtype]}"

    try:
        for s in range(steps):
            if s == w.resize_step:
                cache.resize(w.resize_slots)
                moves = ref.resize(w.resize_slots)
                k2s, sk, ts = cache.tables()
                rk2s, rsk, rts = ref.tables()
                assert np.array_equal(k2s, rk2s) and np.array_equal(sk, rsk) and np.array_equal(ts, rts), \
                    "tables differ after resize"
                report["resize_moves"] = len(moves)
            lg_d = [torch.from_numpy(np.ascontiguousarray(logits[s, l])).to(dev) for l in range(L)]
            xs_h = [W.hidden_states(w, s, l) for l in range(L)]
            xs = [to_act(xs_h[l], w, dev) for l in range(L)]
            refs = {}

            def after_event(l, s=s):
                t = ev_counter[0]
                ridx, rw = orouting.route(logits[s, l], k)
                ev = ref.event(l, ridx)
                refs[l] = (ridx, rw, ev)
                plan = cache.plan(l)
                torch.cuda.synchronize(dev)
                errs = compare_event(plan, ev, idx_d[l].cpu().numpy(), ridx, wt_d[l].cpu().numpy(), rw)
                assert not errs, f"event {t} (step {s}, layer {l}): {errs[:3]}"
                if check_tables_every and t % check_tables_every == 0:
                    k2s, sk, ts = cache.tables()
                    rk2s, rsk, rts = ref.tables()
                    assert np.array_equal(k2s, rk2s), f"event {t}: key_to_slot differs"
                    assert np.array_equal(sk, rsk), f"event {t}: slot_key differs"
                    assert np.array_equal(ts, rts), f"event {t}: slot_ts differs"
                ev_counter[0] += 1

            cache.run_step(lg_d, xs, ys, double_buffer=double_buffer, topk_idx=idx_d, topk_w=wt_d,
                           after_event=after_event)
            cache.synchronize()
            for l in range(L):
                t = refs[l][2].t
                if ffn_every and t % ffn_every == 0:
                    ridx, rw, ev = refs[l]
                    sel = ffn_tokens(l, ridx) if callable(ffn_tokens) else ffn_tokens
                    tok = np.arange(T) if sel is None else np.asarray(sel)
                    yg = ys[l].float().cpu().numpy()[tok]
                    if pool is not None:
                        pending.append((t, pool.submit(oracle_worker.ffn_error_job, w, n_blobs, l, xs_h[l][tok],
                                                       ridx[tok], rw[tok], yg)))
                    else:
                        yr = oracle_ffn(w, bank, n_blobs, l, xs_h[l][tok], ridx[tok], rw[tok])
                        check_ffn(t, *ffn_error(yg, yr))
            if check_slots:  # slots filled this step hold their key's blob, byte for byte
                _, rsk, rts = ref.tables()
                first = refs[0][2].t
                touched = np.flatnonzero(rts >= first)
                for slot in touched[:: max(1, len(touched) // 3)][:4].tolist():
                    key = int(rsk[slot])
                    got = cache.pool[slot * w.expert_bytes:(slot + 1) * w.expert_bytes].cpu().numpy()
                    want = bank_blob(bank, w, n_blobs, key // w.num_experts, key % w.num_experts)
                    assert np.array_equal(got, want), f"step {s}: slot {slot} bytes differ from key {key}'s blob"
                    report["slots_checked"] += 1
        for t, fut in pending:
            check_ffn(t, *fut.result())
        st = cache.stats()
        report["events"] = ev_counter[0]
        report["stats"] = st
        report["miss_rate"] = st["misses"] / max(1, st["unique_experts"])
        assert st["misses"] == ref.n_miss and st["hits"] == ref.n_hit and st["unique_experts"] == ref.n_unique
        assert st["evictions"] == ref.n_evict, (st["evictions"], ref.n_evict)
    finally:
        cache.close()
        if pool is not None:
            pool.shutdown(cancel_futures=True)
    return report


def run_parity_graph(w: W.Workload, steps: int, bank_blobs: int | None = None, double_buffer: bool = True,
                     ffn_every: int = 1, device="cuda:0", timing: bool = False, fetch_mode: int = 1):
    """Replay one captured step graph for `steps` steps and compare every
    layer's plan, the tables after each step, and sampled FFN outputs with the
    oracle (the plans stay readable after the step: each layer keeps its own)."""
    from expert_cache_host_layer_gb300.pipeline import ExpertCache, StepGraph
    dev = torch.device(device)
    bank, n_blobs = make_bank(w, bank_blobs)
    logits = W.router_logits(w.replace(steps=steps))
    cache = ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, w.num_slots,
                        max(w.tokens, 1), bank, n_blobs, fetch_mode=fetch_mode, device=device)
    ref = ExpertCacheOracle(w.num_layers, w.num_experts, w.num_slots)
    L, T, k = w.num_layers, w.tokens, w.top_k
    lg_buf = [torch.empty((T, w.num_experts), dtype=torch.float32, device=dev) for _ in range(L)]
    x_buf = [torch.empty((T, w.hidden), dtype=cache.act_dtype, device=dev) for _ in range(L)]
    y_buf = [torch.empty((T, w.hidden), dtype=torch.float32, device=dev) for _ in range(L)]
    report = {"events": 0, "ffn_checked": 0, "max_err": 0.0}
    graph = StepGraph(cache, lg_buf, x_buf, y_buf, double_buffer, timing=timing)
    try:
        for s in range(steps):
            xs_h = [W.hidden_states(w, s, l) for l in range(L)]
            for l in range(L):
                lg_buf[l].copy_(torch.from_numpy(np.ascontiguousarray(logits[s, l])))
                x_buf[l].copy_(to_act(xs_h[l], w, dev))
            graph.launch()
            cache.synchronize()
            for l in range(L):
                ridx, rw = orouting.route(logits[s, l], k)
                ev = ref.event(l, ridx)
                plan = cache.plan(l)
                errs = compare_event(plan, ev, ridx, ridx, None, rw)
                assert not errs, f"graph step {s}, layer {l}: {errs[:3]}"
                report["events"] += 1
                if ffn_every and ev.t % ffn_every == 0:
                    yr = oracle_ffn(w, bank, n_blobs, l, xs_h[l], ridx, rw)
                    mx, _ = ffn_error(y_buf[l].cpu().numpy(), yr)
                    report["max_err"] = max(report["max_err"], mx)
                    report["ffn_checked"] += 1
                    assert mx <= TOL[w.wdtype], f"graph step {s}, layer {l}: FFN err {mx:.3e}"
            k2s, sk, ts = cache.tables()
            rk2s, rsk, rts = ref.tables()
            assert np.array_equal(k2s, rk2s) and np.array_equal(sk, rsk) and np.array_equal(ts, rts), f"step {s}"
            if timing:
                report["trace"] = graph.trace()
                report["timing"] = graph.timing()
    finally:
        graph.close()
        cache.close()
    return report
