"""Per-step driver over the C ABI: owns the pinned host bank, the device slot
pool and the cache handle, and runs the layer schedule.

Double-buffered schedule of one step (misses of layer l+1 stream in on the
copy stream while layer l's FFN runs - "FreeToken: Efficient Edge-Native MoE
Serving ...", ablation paragraph):

    route(0); fetch(0)
    for l in 0..L-1:  route(l+1); fetch(l+1); forward(l)

Serial schedule (double buffering off): route(l); fetch(l); forward(l).

PyTorch only allocates memory and provides the compute stream; every step of
the path runs in libft's kernels.
"""
from __future__ import annotations

import torch

from . import (FT_FETCH_SM_PULL, FT_W_F32, ft_cache_create, ft_cache_destroy, ft_cache_overhead_bytes,
               ft_host_bank_alloc, ft_host_bank_free,
               ft_cache_resize, ft_expert_bytes, ft_slots_for_budget,
               ft_fetch_misses, ft_get_copy_stream, ft_get_plan, ft_get_stats, ft_get_tables, ft_get_timing,
               ft_moe_forward, ft_reset_stats, ft_route_classify, ft_step_graph_create, ft_step_graph_destroy,
               ft_step_graph_launch, ft_step_graph_timing, ft_step_graph_trace, ft_synchronize, ft_timing_enable,
               make_config)


class ExpertCache:
    """A libft cache with its host bank and device slot pool."""

    def __init__(self, num_layers, num_experts, top_k, hidden, inter, wdtype, num_slots, max_tokens, bank,
                 bank_blobs=None, fetch_mode=FT_FETCH_SM_PULL, pull_ctas=0, copy_streams=1, device="cuda:0",
                 fetch_warps=0,
                 stream: torch.cuda.Stream | None = None):
        self.L, self.E, self.k, self.H, self.I = num_layers, num_experts, top_k, hidden, inter
        self.wdtype = wdtype
        self.eb = ft_expert_bytes(hidden, inter, wdtype)
        if self.eb == 0:
            raise ValueError("unsupported expert shape")
        self.device = torch.device(device)
        self.bank = bank  # torch uint8 tensor in (pinned) host memory, [bank_blobs * expert_bytes]
        self.bank_blobs = bank_blobs or num_layers * num_experts
        self.stream = stream or torch.cuda.current_stream(self.device)
        self.act_dtype = torch.float32 if wdtype == FT_W_F32 else torch.bfloat16  # x
        self.out_dtype = torch.float32                                              # y
        self.pool = torch.empty(num_slots * self.eb, dtype=torch.uint8, device=self.device)
        self.num_slots = num_slots
        cfg = make_config(num_layers, num_experts, top_k, hidden, inter, wdtype, bank.data_ptr(),
                          bank.numel() * bank.element_size(), self.bank_blobs, max_tokens, fetch_mode, pull_ctas,
                          copy_streams, fetch_warps)
        self.cfg = cfg
        self.handle = ft_cache_create(cfg, self.pool.data_ptr(), num_slots, self.stream.cuda_stream)
        self.copy_stream = torch.cuda.ExternalStream(ft_get_copy_stream(self.handle), device=self.device)

    # ---- budget-driven sizing ---------------------------------------------
    @staticmethod
    def slots_for_budget(num_layers, num_experts, top_k, hidden, inter, wdtype, max_tokens, budget_bytes,
                         fetch_mode=FT_FETCH_SM_PULL) -> int:
        """The most slots whose pool plus the library's own device memory fit
        in budget_bytes (ft_slots_for_budget)."""
        cfg = make_config(num_layers, num_experts, top_k, hidden, inter, wdtype, 0, 0, 1, max_tokens, fetch_mode)
        return ft_slots_for_budget(cfg, int(budget_bytes))

    @staticmethod
    def auto_budget(device="cuda:0", reserve_bytes=0) -> int:
        """The free device memory now, minus what the caller keeps for other
        work: the budget of an automatically sized cache."""
        free, _ = torch.cuda.mem_get_info(torch.device(device))
        return max(0, free - int(reserve_bytes))

    @classmethod
    def from_budget(cls, budget_bytes, num_layers, num_experts, top_k, hidden, inter, wdtype, max_tokens, bank,
                    bank_blobs=None, fetch_mode=FT_FETCH_SM_PULL, **kw):
        slots = cls.slots_for_budget(num_layers, num_experts, top_k, hidden, inter, wdtype, max_tokens,
                                     budget_bytes, fetch_mode)
        return cls(num_layers, num_experts, top_k, hidden, inter, wdtype, slots, max_tokens, bank, bank_blobs,
                   fetch_mode=fetch_mode, **kw)

    def device_bytes(self) -> int:
        """Slot pool plus the library's device memory for the current size."""
        return self.num_slots * self.eb + ft_cache_overhead_bytes(self.cfg, self.num_slots)

    def resize_to_budget(self, budget_bytes):
        """Move the cache, at a safe point, to the most slots the new budget
        holds: into a new pool of that size (the old pool is released), so a
        shrink gives the memory back.  Returns the new slot count."""
        slots = ft_slots_for_budget(self.cfg, int(budget_bytes))
        if slots != self.num_slots:
            self.resize(slots, torch.empty(slots * self.eb, dtype=torch.uint8, device=self.device))
        return slots

    # ---- thin wrappers ---------------------------------------------------
    def route_classify(self, layer, logits: torch.Tensor, topk_idx=None, topk_w=None):
        T = logits.shape[0] if logits.dim() == 2 else 0
        ft_route_classify(self.handle, layer, logits.data_ptr() if T else 0, T,
                          topk_idx.data_ptr() if topk_idx is not None else 0,
                          topk_w.data_ptr() if topk_w is not None else 0)

    def fetch_misses(self, layer):
        ft_fetch_misses(self.handle, layer)

    def moe_forward(self, layer, x: torch.Tensor, y: torch.Tensor):
        T = x.shape[0]
        ft_moe_forward(self.handle, layer, x.data_ptr() if T else 0, T, y.data_ptr() if T else 0)

    def resize(self, new_num_slots, new_pool: torch.Tensor | None = None):
        """Safe-point resize; shrinking keeps the same pool (in place) unless new_pool is given."""
        if new_pool is None:
            if new_num_slots <= self.num_slots:
                new_pool = self.pool
            else:
                new_pool = torch.empty(new_num_slots * self.eb, dtype=torch.uint8, device=self.device)
        ft_cache_resize(self.handle, new_pool.data_ptr(), new_num_slots)
        self.pool, self.num_slots = new_pool, new_num_slots

    def synchronize(self):
        ft_synchronize(self.handle)

    def plan(self, layer):
        return ft_get_plan(self.handle, layer, self.E)

    def tables(self):
        return ft_get_tables(self.handle, self.L * self.E, self.num_slots)

    def stats(self):
        return ft_get_stats(self.handle)

    def reset_stats(self):
        ft_reset_stats(self.handle)

    def timing_enable(self, on=True):
        ft_timing_enable(self.handle, on)

    def timing(self):
        return ft_get_timing(self.handle)

    def close(self):
        if self.handle:
            ft_cache_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- one step over all layers ------------------------------------------
    def run_step(self, logits, xs, ys, double_buffer=True, topk_idx=None, topk_w=None, after_event=None):
        """logits[l]: [T,E] f32, xs[l]: [T,H] act_dtype, ys[l]: [T,H] f32 device tensors per layer l.

        `after_event(layer)` (tests) is called right after each layer's
        route_classify is enqueued.
        """
        L = self.L

        def route(l):
            self.route_classify(l, logits[l], None if topk_idx is None else topk_idx[l],
                                None if topk_w is None else topk_w[l])
            if after_event is not None:
                after_event(l)
            self.fetch_misses(l)

        if double_buffer:
            route(0)
            for l in range(L):
                if l + 1 < L:
                    route(l + 1)
                self.moe_forward(l, xs[l], ys[l])
        else:
            for l in range(L):
                route(l)
                self.moe_forward(l, xs[l], ys[l])


class StepGraph:
    """One captured step over all layers (see ft_step_graph_create); the
    logits/x/y tensors are the fixed buffers the graph reads and writes."""

    def __init__(self, cache: ExpertCache, logits, xs, ys, double_buffer=True, timing=False):
        self.cache = cache
        self.logits, self.xs, self.ys = logits, xs, ys  # keep the buffers alive
        T = logits[0].shape[0]
        self.handle = ft_step_graph_create(cache.handle, [t.data_ptr() for t in logits], [t.data_ptr() for t in xs],
                                           [t.data_ptr() for t in ys], T, double_buffer, timing)

    def launch(self):
        ft_step_graph_launch(self.handle)

    def timing(self):
        return ft_step_graph_timing(self.handle, self.cache.L)

    def trace(self):
        return ft_step_graph_trace(self.handle, self.cache.L)

    def close(self):
        if self.handle:
            ft_step_graph_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pinned_bank(nbytes: int) -> torch.Tensor:
    """A pinned, device-mapped host byte buffer of exactly nbytes for the
    expert bank (ft_host_bank_alloc), as a CPU uint8 tensor that frees the
    memory when the last view of it is gone.  (PyTorch's own pinned allocator
    rounds a request up to a power of two: a 64.4 GB bank would pin 128 GB.)"""
    import ctypes
    import weakref

    import numpy as np
    ptr = ft_host_bank_alloc(nbytes)
    raw = (ctypes.c_uint8 * nbytes).from_address(ptr)
    weakref.finalize(raw, _free_bank, ptr)
    return torch.from_numpy(np.ctypeslib.as_array(raw))


def _free_bank(ptr: int):
    try:
        ft_host_bank_free(ptr)
    except Exception:  # at interpreter exit the runtime may already be gone; the OS reclaims the memory
        pass
