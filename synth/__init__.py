"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

This package makes inputs only (router logits, hidden states, expert weight
blobs in the runtime layout); it computes no step of the expert-cache method.
Every value comes from the counter-based SplitMix64 generator in ``synth.c``,
compiled on first use into ``_build/libsynth.so`` next to it.

Workload recipes (shapes, value distributions, routing structure) follow the
pages' workloads: Qwen3.6-35B-A3B-shaped layers (256 experts, top-8,
hidden 2048, expert intermediate 512) and DeepSeek-V4-Flash-shaped layers
(256 experts, top-8, hidden 4096, intermediate 2048, fp8 block-scaled).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
# SYNTH_SANITIZE=1: a build with AddressSanitizer and UndefinedBehaviorSanitizer
# (the process must preload the ASan runtime), for the host-sanitizer test
_SANITIZE = os.environ.get("SYNTH_SANITIZE", "") == "1"
_OUT_DIR = os.path.join(_HERE, "_build_san" if _SANITIZE else "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsynth.so")
_SAN_FLAGS = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-g"]
_lock = threading.Lock()
_lib = None

BASE_SEED = 20261202
W_F32, W_BF16, W_FP8 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile synth.c into _build/libsynth.so (gcc, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O3", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                               *(_SAN_FLAGS if _SANITIZE else []), "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i32, i64, f32, f64, p = (ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                          ctypes.c_double, ctypes.c_void_p)
            sig = {
                "synth_key": (u64, [u64, u64, u64, u64, u64]),
                "synth_u64": (u64, [u64, u64]),
                "synth_e4m3_encode": (ctypes.c_uint8, [f32]),
                "synth_bf16_encode": (ctypes.c_uint16, [f32]),
                "synth_f32_to_bf16": (None, [p, p, i64]),
                "synth_bf16_to_f32": (None, [p, p, i64]),
                "synth_normal_f32": (None, [u64, u64, i64, f32, p, i32]),
                "synth_expert_bytes": (i64, [i32, i32, i32]),
                "synth_expert_blobs": (i32, [u64, i32, i32, i32, p, i64, p, i32]),
                "synth_zipf_bias": (None, [u64, i32, i32, f64, p]),
                "synth_router_decode": (None, [u64, i32, i32, i32, i32, i32, f64, f64, f32, p]),
                "synth_router_iid": (None, [u64, i32, i32, i32, i32, f64, p, i32]),
                "synth_router_ties": (None, [u64, i32, i64, p]),
                "synth_hidden": (None, [u64, i32, i32, i32, i32, i32, i32, p, i32]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def threads() -> int:
    """Generator threads: SYNTH_THREADS if set (worker processes use 1), else the host's cores."""
    env = os.environ.get("SYNTH_THREADS")
    if env:
        return max(1, min(64, int(env)))
    return max(1, min(64, os.cpu_count() or 1))


# ---- scalar helpers ----------------------------------------------------------

def key(seed: int, a: int = 0, b: int = 0, c: int = 0, d: int = 0) -> int:
    return int(_L().synth_key(seed, a, b, c, d))


def u64(k: int, n: int) -> int:
    return int(_L().synth_u64(k, n))


def e4m3_encode(x: float) -> int:
    return int(_L().synth_e4m3_encode(x))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _L().synth_f32_to_bf16(_ptr(x), _ptr(out), x.size)
    return out


def bf16_values(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _L().synth_bf16_to_f32(_ptr(bits), _ptr(out), bits.size)
    return out


# ---- arrays --------------------------------------------------------------------

def normal(k: int, n: int, scale: float = 1.0, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _L().synth_normal_f32(k, start, n, scale, _ptr(out), threads())
    return out


def expert_bytes(hidden: int, inter: int, wdtype: int) -> int:
    return int(_L().synth_expert_bytes(hidden, inter, wdtype))


def expert_blobs(seed: int, hidden: int, inter: int, wdtype: int, blob_ids, out: np.ndarray | None = None,
                 out_ptr: int | None = None) -> np.ndarray | None:
    """Generate the expert blobs `blob_ids` (runtime layout) consecutively.

    Writes into `out` (uint8, len(blob_ids) * expert_bytes) or into raw memory
    at `out_ptr` (for example a pinned host buffer); returns the array when one
    was allocated here.
    """
    ids = np.ascontiguousarray(np.asarray(blob_ids, dtype=np.int64))
    eb = expert_bytes(hidden, inter, wdtype)
    if eb <= 0:
        raise ValueError("unsupported expert shape / dtype")
    if out_ptr is None:
        if out is None:
            out = np.empty(ids.size * eb, dtype=np.uint8)
        assert out.nbytes >= ids.size * eb
        out_ptr = _ptr(out)
    rc = _L().synth_expert_blobs(seed, hidden, inter, wdtype, _ptr(ids), ids.size, out_ptr, threads())
    if rc != 0:
        raise RuntimeError("synth_expert_blobs failed")
    return out


def zipf_bias(seed: int, layer: int, E: int, a: float = 1.1) -> np.ndarray:
    out = np.empty(E, dtype=np.float32)
    _L().synth_zipf_bias(seed, layer, E, a, _ptr(out))
    return out


def router_decode(seed: int, stream: int, L: int, E: int, k: int, steps: int, zipf_a: float = 1.1,
                  p_keep: float = 0.7, lift: float = 32.0) -> np.ndarray:
    """Correlated decode routing logits of one stream: float32 [steps][L][E]."""
    if k > 64:
        raise ValueError("k > 64 not supported by the generator")
    out = np.empty((steps, L, E), dtype=np.float32)
    _L().synth_router_decode(seed, stream, L, E, k, steps, zipf_a, p_keep, lift, _ptr(out))
    return out


def router_iid(seed: int, stream: int, layer: int, T: int, E: int, zipf_a: float = 1.1) -> np.ndarray:
    """i.i.d. N(0,1) + Zipf bias logits for one chunk at one layer: float32 [T][E]."""
    out = np.empty((T, E), dtype=np.float32)
    _L().synth_router_iid(seed, stream, layer, T, E, zipf_a, _ptr(out), threads())
    return out


def router_ties(seed: int, stream: int, shape) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _L().synth_router_ties(seed, stream, out.size, _ptr(out))
    return out


def hidden(seed: int, stream: int, step: int, layer: int, T: int, H: int, round_bf16: bool) -> np.ndarray:
    """Hidden states x [T][H] ~ N(0,1) (float32 values, bf16-exact when round_bf16)."""
    out = np.empty((T, H), dtype=np.float32)
    _L().synth_hidden(seed, stream, step, layer, T, H, int(bool(round_bf16)), _ptr(out), threads())
    return out
