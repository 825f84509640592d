"""Python binding of libft (include/ft.h): argument marshalling only.

Every function here has the name of the C entry point it calls and passes
plain pointers and sizes through ctypes; all work happens in the CUDA
library.  PyTorch (when used) only provides device memory and streams: pass
``tensor.data_ptr()`` and ``stream.cuda_stream``.

Importing this package loads ``_build/libft.so`` (with FT_CHECKED=1 in the
environment, the bounds-checked build ``_build_checked/libft.so``).  If it was
not built, the import fails with an error saying how to build it: there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
CHECKED = os.environ.get("FT_CHECKED", "") == "1"
SANITIZED = os.environ.get("FT_SANITIZE", "") == "1"  # the host code built with UndefinedBehaviorSanitizer
LIB_PATH = os.path.join(_HERE, "_build_checked" if CHECKED else "_build_ubsan" if SANITIZED else "_build", "libft.so")

FT_OK, FT_ERR_INVALID_ARG, FT_ERR_CUDA, FT_ERR_OOM, FT_ERR_CAPACITY, FT_ERR_STATE, FT_ERR_TIMEOUT, \
    FT_ERR_CHECKED, FT_ERR_UNSUPPORTED = range(9)
FT_W_F32, FT_W_BF16, FT_W_FP8E4M3_B128 = 0, 1, 2
FT_FETCH_COPY_ENGINE, FT_FETCH_SM_PULL = 0, 1


class FtError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: {_status_name(status)}: {message}")


class ft_cache_config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("wdtype", ctypes.c_int32),
                ("host_bank", ctypes.c_void_p), ("host_bank_bytes", ctypes.c_uint64),
                ("bank_blobs", ctypes.c_int64), ("max_tokens", ctypes.c_int32), ("fetch_mode", ctypes.c_int32),
                ("pull_ctas", ctypes.c_int32), ("copy_streams", ctypes.c_int32), ("fetch_warps", ctypes.c_int32)]


class ft_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("events", "unique_experts", "hits", "misses", "evictions",
                                              "bytes_fetched", "kernel_launches", "memcpy_calls")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class ft_timing(ctypes.Structure):
    _fields_ = [("route_ms", ctypes.c_double), ("route_n", ctypes.c_int64),
                ("fetch_ms", ctypes.c_double), ("fetch_n", ctypes.c_int64),
                ("ffn_ms", ctypes.c_double), ("ffn_n", ctypes.c_int64),
                ("gemm1_ms", ctypes.c_double), ("gemm1_n", ctypes.c_int64),
                ("gemm2_ms", ctypes.c_double), ("gemm2_n", ctypes.c_int64)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class ft_plan_info(ctypes.Structure):
    _fields_ = [("event", ctypes.c_int32), ("n_tokens", ctypes.c_int32), ("n_unique", ctypes.c_int32),
                ("n_miss", ctypes.c_int32)]


# ---------------------------------------------------------------- loading

def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libft is not built ({LIB_PATH} missing); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` or "
                          "`python expert_cache_host_layer_gb300/build.py" + (" --checked`" if CHECKED else "`"))
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, U8P = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(ctypes.c_uint8)
    st = ctypes.c_int
    sig = {
        "ft_expert_bytes": (ctypes.c_size_t, [I32, I32, I32]),
        "ft_cache_create": (st, [ctypes.POINTER(ft_cache_config), P, I64, P, ctypes.POINTER(P)]),
        "ft_cache_overhead_bytes": (ctypes.c_uint64, [ctypes.POINTER(ft_cache_config), I64]),
        "ft_slots_for_budget": (st, [ctypes.POINTER(ft_cache_config), ctypes.c_uint64, ctypes.POINTER(I64)]),
        "ft_cache_destroy": (st, [P]),
        "ft_cache_resize": (st, [P, P, I64]),
        "ft_route_classify": (st, [P, I32, P, I32, P, P]),
        "ft_fetch_misses": (st, [P, I32]),
        "ft_moe_forward": (st, [P, I32, P, I32, P]),
        "ft_synchronize": (st, [P]),
        "ft_get_plan": (st, [P, I32, ctypes.POINTER(ft_plan_info), P, P, P, P, P, P]),
        "ft_get_tables": (st, [P, P, P, P]),
        "ft_get_stats": (st, [P, ctypes.POINTER(ft_stats)]),
        "ft_reset_stats": (st, [P]),
        "ft_get_pool": (st, [P, ctypes.POINTER(P), ctypes.POINTER(I64)]),
        "ft_get_copy_stream": (st, [P, ctypes.POINTER(P)]),
        "ft_debug_pause_copies": (st, [P, I32]),
        "ft_checked_build": (I32, []),
        "ft_host_bank_alloc": (st, [ctypes.c_uint64, ctypes.POINTER(P)]),
        "ft_host_bank_free": (st, [P]),
        "ft_debug_set_key_slot": (st, [P, I32, I32]),
        "ft_timing_enable": (st, [P, I32]),
        "ft_get_timing": (st, [P, ctypes.POINTER(ft_timing)]),
        "ft_step_graph_create": (st, [P, P, P, P, I32, I32, I32, ctypes.POINTER(P)]),
        "ft_step_graph_launch": (st, [P]),
        "ft_step_graph_timing": (st, [P, P, P, P, P]),
        "ft_step_graph_trace": (st, [P, P]),
        "ft_step_graph_destroy": (st, [P]),
        "ft_moe_decode_ffn_static": (st, [I32, I32, I32, I32, I32, P, I64, P, P, P, P, I32, P, P]),
        "ft_moe_decode_ffn_static_status": (st, [P]),
        "ft_status_str": (ctypes.c_char_p, [st]),
        "ft_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    del U8P
    return lib


_lib = _load()


def _status_name(s: int) -> str:
    return _lib.ft_status_str(s).decode()


def _check(status: int, where: str):
    if status != FT_OK:
        raise FtError(status, where, _lib.ft_last_error().decode())


def library():
    """The loaded ctypes library (exported symbols: see include/ft.h)."""
    return _lib


# ---------------------------------------------------------------- entry points

def ft_expert_bytes(hidden: int, inter: int, wdtype: int) -> int:
    return int(_lib.ft_expert_bytes(hidden, inter, wdtype))


def ft_cache_overhead_bytes(cfg: ft_cache_config, num_slots: int) -> int:
    return int(_lib.ft_cache_overhead_bytes(ctypes.byref(cfg), num_slots))


def ft_slots_for_budget(cfg: ft_cache_config, budget_bytes: int) -> int:
    n = ctypes.c_int64()
    _check(_lib.ft_slots_for_budget(ctypes.byref(cfg), budget_bytes, ctypes.byref(n)), "ft_slots_for_budget")
    return n.value


def ft_cache_create(cfg: ft_cache_config, slot_pool: int, num_slots: int, compute_stream: int = 0) -> int:
    out = ctypes.c_void_p()
    _check(_lib.ft_cache_create(ctypes.byref(cfg), slot_pool, num_slots, compute_stream or None,
                                ctypes.byref(out)), "ft_cache_create")
    return out.value


def ft_cache_destroy(cache: int):
    _check(_lib.ft_cache_destroy(cache), "ft_cache_destroy")


def ft_cache_resize(cache: int, new_pool: int, new_num_slots: int):
    _check(_lib.ft_cache_resize(cache, new_pool, new_num_slots), "ft_cache_resize")


def ft_route_classify(cache: int, layer: int, logits: int, T: int, topk_idx: int = 0, topk_w: int = 0):
    _check(_lib.ft_route_classify(cache, layer, logits or None, T, topk_idx or None, topk_w or None),
           "ft_route_classify")


def ft_fetch_misses(cache: int, layer: int):
    _check(_lib.ft_fetch_misses(cache, layer), "ft_fetch_misses")


def ft_moe_forward(cache: int, layer: int, x: int, T: int, y: int):
    _check(_lib.ft_moe_forward(cache, layer, x or None, T, y or None), "ft_moe_forward")


def ft_synchronize(cache: int):
    _check(_lib.ft_synchronize(cache), "ft_synchronize")


def ft_get_plan(cache: int, layer: int, num_experts: int):
    """The layer's plan as a dict of numpy arrays (synchronous)."""
    import numpy as np
    info = ft_plan_info()
    arrs = {n: np.zeros(num_experts, dtype=np.int32) for n in
            ("unique_expert", "unique_slot", "miss_expert", "miss_slot", "evicted_key")}
    hit = np.zeros(num_experts, dtype=np.uint8)
    _check(_lib.ft_get_plan(cache, layer, ctypes.byref(info), arrs["unique_expert"].ctypes.data,
                            arrs["unique_slot"].ctypes.data, hit.ctypes.data, arrs["miss_expert"].ctypes.data,
                            arrs["miss_slot"].ctypes.data, arrs["evicted_key"].ctypes.data), "ft_get_plan")
    nu, nm = info.n_unique, info.n_miss
    return {"event": info.event, "n_tokens": info.n_tokens, "unique": arrs["unique_expert"][:nu],
            "unique_slot": arrs["unique_slot"][:nu], "hit": hit[:nu], "miss_expert": arrs["miss_expert"][:nm],
            "miss_slot": arrs["miss_slot"][:nm], "evicted_key": arrs["evicted_key"][:nm]}


def ft_get_tables(cache: int, num_keys: int, num_slots: int):
    import numpy as np
    k2s = np.zeros(num_keys, dtype=np.int32)
    sk = np.zeros(num_slots, dtype=np.int32)
    ts = np.zeros(num_slots, dtype=np.int32)
    _check(_lib.ft_get_tables(cache, k2s.ctypes.data, sk.ctypes.data, ts.ctypes.data), "ft_get_tables")
    return k2s, sk, ts


def ft_get_stats(cache: int) -> dict:
    s = ft_stats()
    _check(_lib.ft_get_stats(cache, ctypes.byref(s)), "ft_get_stats")
    return s.as_dict()


def ft_reset_stats(cache: int):
    _check(_lib.ft_reset_stats(cache), "ft_reset_stats")


def ft_get_pool(cache: int):
    p, n = ctypes.c_void_p(), ctypes.c_int64()
    _check(_lib.ft_get_pool(cache, ctypes.byref(p), ctypes.byref(n)), "ft_get_pool")
    return p.value, n.value


def ft_get_copy_stream(cache: int) -> int:
    p = ctypes.c_void_p()
    _check(_lib.ft_get_copy_stream(cache, ctypes.byref(p)), "ft_get_copy_stream")
    return p.value or 0


def ft_debug_pause_copies(cache: int, paused: bool):
    _check(_lib.ft_debug_pause_copies(cache, int(bool(paused))), "ft_debug_pause_copies")


def ft_host_bank_alloc(nbytes: int) -> int:
    p = ctypes.c_void_p()
    _check(_lib.ft_host_bank_alloc(int(nbytes), ctypes.byref(p)), "ft_host_bank_alloc")
    return int(p.value)


def ft_host_bank_free(host: int):
    _check(_lib.ft_host_bank_free(host), "ft_host_bank_free")


def ft_checked_build() -> bool:
    return bool(_lib.ft_checked_build())


def ft_debug_set_key_slot(cache: int, key: int, slot: int):
    _check(_lib.ft_debug_set_key_slot(cache, int(key), int(slot)), "ft_debug_set_key_slot")


def ft_timing_enable(cache: int, on: bool):
    _check(_lib.ft_timing_enable(cache, int(bool(on))), "ft_timing_enable")


def ft_get_timing(cache: int) -> dict:
    t = ft_timing()
    _check(_lib.ft_get_timing(cache, ctypes.byref(t)), "ft_get_timing")
    return t.as_dict()


def make_config(num_layers, num_experts, top_k, hidden, inter, wdtype, host_bank_ptr, host_bank_bytes, bank_blobs,
                max_tokens, fetch_mode=FT_FETCH_SM_PULL, pull_ctas=0, copy_streams=1,
                fetch_warps=0) -> ft_cache_config:
    return ft_cache_config(num_layers, num_experts, top_k, hidden, inter, wdtype, host_bank_ptr, host_bank_bytes,
                           bank_blobs, max_tokens, fetch_mode, pull_ctas, copy_streams, fetch_warps)


def ft_step_graph_create(cache: int, logits_ptrs, x_ptrs, y_ptrs, T: int, double_buffer: bool = True,
                         timing: bool = False) -> int:
    """Capture one step over all layers into a CUDA graph; pointer lists hold one buffer per layer."""
    arr = ctypes.c_void_p * len(logits_ptrs)
    out = ctypes.c_void_p()
    _check(_lib.ft_step_graph_create(cache, arr(*logits_ptrs), arr(*x_ptrs), arr(*y_ptrs), T, int(bool(double_buffer)),
                                     int(bool(timing)), ctypes.byref(out)), "ft_step_graph_create")
    return out.value


def ft_step_graph_launch(graph: int):
    _check(_lib.ft_step_graph_launch(graph), "ft_step_graph_launch")


def ft_step_graph_timing(graph: int, num_layers: int):
    """(route_ms[L], fetch_ms[L], ffn_ms[L], step_ms) of the graph's last launch (waits for it)."""
    import numpy as np
    r = np.zeros(num_layers, dtype=np.float64)
    fe = np.zeros(num_layers, dtype=np.float64)
    f = np.zeros(num_layers, dtype=np.float64)
    st = ctypes.c_double()
    _check(_lib.ft_step_graph_timing(graph, r.ctypes.data, fe.ctypes.data, f.ctypes.data, ctypes.byref(st)),
           "ft_step_graph_timing")
    return r, fe, f, st.value


def ft_step_graph_trace(graph: int, num_layers: int):
    """[L][6] ms from the step start: route, fetch, FFN begin/end per layer (last launch)."""
    import numpy as np
    t = np.zeros(6 * num_layers, dtype=np.float64)
    _check(_lib.ft_step_graph_trace(graph, t.ctypes.data), "ft_step_graph_trace")
    return t.reshape(num_layers, 6)


def ft_step_graph_destroy(graph: int):
    _check(_lib.ft_step_graph_destroy(graph), "ft_step_graph_destroy")


def ft_moe_decode_ffn_static(hidden: int, inter: int, wdtype: int, num_experts: int, top_k: int, slot_pool: int,
                             num_slots: int, expert_slot: int, topk_idx: int, topk_w: int, x: int, T: int, y: int,
                             stream: int = 0):
    """Decode FFN whose working memory is a static device array (no allocation)."""
    _check(_lib.ft_moe_decode_ffn_static(hidden, inter, wdtype, num_experts, top_k, slot_pool or None, num_slots,
                                         expert_slot or None, topk_idx or None, topk_w or None, x or None, T,
                                         y or None, stream or None), "ft_moe_decode_ffn_static")


def ft_moe_decode_ffn_static_status(stream: int = 0):
    """Raise FtError if an earlier static-scratch FFN call hit a bounded-wait timeout (clears it)."""
    _check(_lib.ft_moe_decode_ffn_static_status(stream or None), "ft_moe_decode_ffn_static_status")


def ft_status_str(status: int) -> str:
    return _status_name(status)


def ft_last_error() -> str:
    return _lib.ft_last_error().decode()
