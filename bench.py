"""Benchmark of the per-MoE-layer hot path on GB300.

One step = one decode token through all 40 MoE layers of the
Qwen3.6-35B-A3B-shaped workload (256 experts, top-8, hidden 2048,
intermediate 512, bf16 experts, full 64.4 GB bank pinned in host memory,
3072-slot GPU cache = 30% of the bank, correlated Zipf routing): per layer
route_classify (top-k, dedup, hit/miss, LRU victims), the miss fetch on the
copy stream one layer ahead, and the expert FFN reading the slots.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica (the path has no data-parallel exchange): value = all ranks' tokens /
the slowest rank's time.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import workloads as W  # noqa: E402

METRIC = "MoE decode tokens/s (35B-A3B shape, 1 GB300); expert-GEMM HBM GB/s; miss rate"
L2_BYTES = 129 * 1024 * 1024


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=8)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=W.QWEN35B_DECODE.name, choices=sorted(W.ALL))
    p.add_argument("--fetch-mode", type=int, default=1, help="0 copy engine, 1 SM pull")
    p.add_argument("--pull-ctas", type=int, default=0)
    p.add_argument("--copy-streams", type=int, default=1)
    p.add_argument("--fetch-warps", type=int, default=0, help="SM pull: FFN warps per SM copying the next misses")
    p.add_argument("--serial", action="store_true", help="double buffering off")
    p.add_argument("--bank-blobs", type=int, default=0, help="0 = full bank; fewer = aliased bank")
    p.add_argument("--slots", type=int, default=0, help="override the cache size")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-link", action="store_true")
    p.add_argument("--trace", action="store_true", help="print one step's per-layer timeline to stderr")
    p.add_argument("--ffn-only", action="store_true",
                   help="only time the decode FFN kernel with every expert a hit (no fetch) and print it")
    p.add_argument("--prefill-gemm-only", action="store_true",
                   help="only time the prefill chunk's two tensor-core GEMMs (all hits, no fetch) and print them")
    p.add_argument("--gemm-experts", type=int, default=0,
                   help="--prefill-gemm-only: fewer experts (a small case for profiling)")
    p.add_argument("--gemm-tokens", type=int, default=0,
                   help="--prefill-gemm-only: fewer tokens (a small case for profiling)")
    p.add_argument("--cpu-steps", type=int, default=2,
                   help="reference arm: decode steps of the oracle sample timed per step")
    p.add_argument("--cpu-baseline-steps", type=int, default=8,
                   help="decode steps of the oracle sample behind cpu_baseline")
    p.add_argument("--no-blocks", action="store_true",
                   help="skip the 4/8-stream, prefill and fp8 blocks (the headline decode only)")
    p.add_argument("--timing-steps", type=int, default=32,
                   help="steps of the timing pass (graphs with event nodes around every kernel)")
    return p.parse_args()


# --------------------------------------------------------------------- helpers

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


def measured_bf16_tflops() -> float:
    """Burst bf16 dense TFLOP/s from MEASURED_PEAKS.json (the recipe's fallback
    1900 if absent): the denominator of the prefill GEMMs' tensor fraction."""
    try:
        with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------- oracle arm

def _oracle_ffn_job(w, layer, x, idx, gates):
    """One layer event's oracle FFN in a worker process: the unique experts'
    blobs are generated first (input preparation, not timed), then the
    dequantisation and the fp64 SwiGLU FFN are timed.  Returns (pid, s)."""
    from oracle import ffn as offn
    uniq = sorted({int(v) for v in np.asarray(idx).ravel()})
    raw = {e: synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, [w.blob_of(layer, e)]) for e in uniq}
    t0 = time.perf_counter()
    blobs = {e: offn.dequant_blob(b, w.hidden, w.inter, w.wdtype) for e, b in raw.items()}
    offn.moe_ffn(x, idx, gates, lambda e: blobs[e])
    return os.getpid(), time.perf_counter() - t0


def oracle_sample(w: W.Workload, steps: int, workers: int, logits=None):
    """The CPU oracle on the first `steps` decode steps of workload w: routing
    and the LRU cache simulation run in order on one host thread (they are a
    sequential decision stream); the FFN of every layer event runs in a pool
    of `workers` spawned processes.  Oracle time = the decision stream's time
    + the busiest worker's FFN time.  Returns (tokens/s, oracle seconds, CPU
    seconds summed over the thread and the workers)."""
    import concurrent.futures
    import multiprocessing

    from oracle import routing as orouting
    from oracle.cache import ExpertCacheOracle
    if logits is None:
        logits = W.router_logits(w.replace(steps=steps))
    ref = ExpertCacheOracle(w.num_layers, w.num_experts, w.num_slots)
    t_dec = 0.0
    busy = {}
    # one thread per worker process: no BLAS or generator thread pools on top of the
    # processes (the executor spawns its workers lazily, so the variables stay set
    # for the pool's whole life)
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                                              "SYNTH_THREADS")}
    os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1", SYNTH_THREADS="1")
    try:
        with concurrent.futures.ProcessPoolExecutor(workers,
                                                    mp_context=multiprocessing.get_context("spawn")) as pool:
            futs = []
            for s in range(steps):
                for l in range(w.num_layers):
                    t0 = time.perf_counter()
                    idx, gw = orouting.route(logits[s, l], w.top_k)
                    ref.event(l, idx)
                    t_dec += time.perf_counter() - t0
                    futs.append(pool.submit(_oracle_ffn_job, w, l, W.hidden_states(w, s, l), idx, gw))
            for f in futs:
                pid, dt = f.result()
                busy[pid] = busy.get(pid, 0.0) + dt
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    spent = t_dec + max(busy.values())
    return steps * w.tokens / spent, spent, t_dec + sum(busy.values())


def cpu_workers() -> int:
    return max(1, os.cpu_count() or 1)


def cpu_baseline(w: W.Workload, steps: int):
    workers = cpu_workers()
    v, dt, cpu_s = oracle_sample(w, steps, workers)
    return {"value": v, "unit": "tokens/s", "cores": workers, "kind": "oracle",
            "sample": f"first {steps} decode steps x {w.num_layers} layers of {w.name} (cold cache): routing and "
                      f"LRU simulation in order on one thread, fp64 SwiGLU FFN of each layer event over "
                      f"{workers} worker processes; {dt:.1f} s of oracle time (decisions + busiest worker), "
                      f"{cpu_s:.1f} CPU-seconds in all"}


def workload_config(w: W.Workload, world: int, n_blobs: int) -> dict:
    """The `config` block both arms print for the same workload."""
    return {"workload": w.name, "global_batch": world * w.tokens, "layers": w.num_layers,
            "experts": w.num_experts, "top_k": w.top_k, "hidden": w.hidden, "inter": w.inter,
            "slots": w.num_slots, "bank_blobs": n_blobs, "bank_gb": round(n_blobs * w.expert_bytes / 1e9, 2),
            "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2 (each step reads ~2 GB of expert slots)"}


def run_reference(args, w):
    rank, _, world = dist_setup(args.gpus)
    if rank != 0:
        return
    if args.slots:
        w = w.replace(num_slots=args.slots)
    # each step: the oracle over a bounded sample (the first decode steps of
    # the same workload, cold cache), all host cores
    workers = cpu_workers()
    logits = W.router_logits(w.replace(steps=args.cpu_steps))
    per = []
    for i in range(args.warmup + args.steps):
        v, dt, _ = oracle_sample(w, args.cpu_steps, workers, logits)
        if i >= args.warmup:
            per.append(dt / args.cpu_steps)
    ms = 1e3 * statistics.mean(per)
    value = w.tokens / (ms / 1e3)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.gpus, args.bank_blobs or w.blobs),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": workers, "kind": "oracle",
                             "sample": f"each step: the first {args.cpu_steps} decode steps (cold cache) of "
                                       f"{w.name}; decisions on one thread, FFN over {workers} worker processes"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- our arm

# dram__bytes_read.sum + dram__bytes_write.sum of ffn_fused_kernel launches from ncu captures, keyed by
# workload; they belong to the kernel as captured: drop an entry whenever that kernel changes.
# The all-hit launches of --ffn-only, per launch (an ncu --set full capture of two launches).
FFN_ONLY_TRAFFIC_PER_LAUNCH = {"qwen35b-a3b-shape-decode-b1": (50.393856e6 + 1.28e3 + 50.3936e6 + 1.024e3) / 2}
# The in-pipeline launches (copies riding along) of a small case of the same kernel, whose device memory
# fits a capture (320 slots, a 640-blob bank; 6 launches of the same kernel instantiation):
# DRAM bytes read per unique expert, and DRAM bytes written per launch.  The blobs a launch copies in land
# in the 129 MB L2 and reach DRAM after the launch, so its own writes are near zero; the reads scale with
# the unique experts, which the full workload's traffic is scaled by.
FFN_PIPELINE_TRAFFIC = {"qwen35b-a3b-shape-decode-b1": ((50.396e6 + 50.396e6 + 50.395e6 + 50.397e6 + 50.404e6
                                                          + 50.404e6) / 6 / 8, (43e3 + 25e3 + 19e3) / 6)}


def pipeline_traffic(name: str, mean_unique: float):
    """DRAM bytes per in-pipeline FFN launch scaled from the small capture, or None."""
    c = FFN_PIPELINE_TRAFFIC.get(name)
    return None if c is None else c[0] * mean_unique + c[1]


def prefill_measure(dev, peak_tflops, steps=2):
    """The 35B-shaped prefill chunk (16,384 tokens per layer, 40 layers, 3072
    slots): 40 x ~214 unique experts per step thrash the 3072-slot LRU, so
    every step fetches nearly all its experts over the host link.  One step's
    routing and hidden states are replayed `steps` times through a captured
    step graph (the first as warm-up); the bank is aliased to 1024 blobs
    (same transfer sizes).  Returns per-layer phase times and throughput."""
    import torch

    from expert_cache_host_layer_gb300.pipeline import ExpertCache, StepGraph
    w = W.QWEN35B_PREFILL
    L, T = w.num_layers, w.tokens
    n_blobs = 1024
    from expert_cache_host_layer_gb300.pipeline import pinned_bank
    bank = pinned_bank(n_blobs * w.expert_bytes)
    synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, np.arange(n_blobs), out_ptr=bank.data_ptr())
    bank_warm(w, dev, bank, n_blobs)
    lg = [torch.from_numpy(synth.router_iid(w.seed, 0, l, T, w.num_experts, 1.1)).to(dev) for l in range(L)]
    xs = [torch.from_numpy(W.hidden_states(w, 0, l)).to(dev, torch.bfloat16) for l in range(L)]
    ys = [torch.empty((T, w.hidden), dtype=torch.float32, device=dev) for _ in range(L)]
    c = ExpertCache(L, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, w.num_slots, T, bank, n_blobs,
                    fetch_mode=1, device=dev)
    out = {}
    try:
        for double in (True, False):
            g = StepGraph(c, lg, xs, ys, double, timing=True)
            try:
                g.launch()  # warm-up step
                c.synchronize()
                st0 = c.stats()
                tot = {"route": 0.0, "fetch": 0.0, "ffn": 0.0, "step": 0.0}
                for _ in range(steps - 1):
                    g.launch()
                    r, fe, f, step_ms = g.timing()
                    tot["route"] += r.sum(); tot["fetch"] += fe.sum(); tot["ffn"] += f.sum(); tot["step"] += step_ms
                st1 = c.stats()
            finally:
                g.close()
            n = max(1, steps - 1)
            rows = T * w.top_k
            flop = 2.0 * rows * (2 * w.inter * w.hidden + w.hidden * w.inter)  # per layer
            ffn_ms = tot["ffn"] / n / L
            out["double_buffer" if double else "serial"] = {
                "tokens_per_s": T / (tot["step"] / n / 1e3), "ms_per_step": tot["step"] / n,
                "per_layer_ms": {k: tot[k] / n / L for k in ("route", "fetch", "ffn")},
                "ffn_tflops": flop / (ffn_ms / 1e3) / 1e12,
                "tensor_frac": flop / (ffn_ms / 1e3) / 1e12 / peak_tflops,
                "fetched_gb_per_step": (st1["bytes_fetched"] - st0["bytes_fetched"]) / n / 1e9,
                "miss_rate": (st1["misses"] - st0["misses"]) / max(1, st1["unique_experts"] - st0["unique_experts"])}
    finally:
        c.close()
    out["note"] = ("step graph with timing event nodes, 40 layers, one 16,384-token chunk each; FFN = grouping, "
                   "permutation, the two tcgen05 grouped GEMMs (gate/up + SwiGLU, down) and the combine; times "
                   "from the event nodes")
    return out


def prefill_gemm_only(dev, peak_tflops, reps=6, w=None):
    """The prefill chunk's two tensor-core GEMMs alone, through the public
    API: a one-layer cache of 512 slots routes the same 16,384-token chunk
    every event, so after the first event every unique expert hits and no
    fetch runs beside the GEMMs.  The library's event timing brackets the
    gate/up + SwiGLU GEMM and the down GEMM of each forward.  The weights the
    GEMMs stream (~214 experts x 6.3 MB) are larger than L2."""
    import torch

    from expert_cache_host_layer_gb300.pipeline import ExpertCache, pinned_bank
    w = w or W.QWEN35B_PREFILL
    T, E, k = w.tokens, w.num_experts, w.top_k
    bank = pinned_bank(E * w.expert_bytes)
    synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, np.arange(E), out_ptr=bank.data_ptr())
    lg = torch.from_numpy(synth.router_iid(w.seed, 0, 0, T, E, 1.1)).to(dev)
    x = torch.from_numpy(W.hidden_states(w, 0, 0)).to(dev, torch.bfloat16)
    y = torch.empty((T, w.hidden), dtype=torch.float32, device=dev)
    c = ExpertCache(1, E, k, w.hidden, w.inter, w.wdtype, 2 * E, T, bank, E, fetch_mode=1, device=dev)
    try:
        def event():
            c.route_classify(0, lg)
            c.fetch_misses(0)
            c.moe_forward(0, x, y)
        for _ in range(2):  # fill, then one all-hit warm-up
            event()
        c.synchronize()
        st0 = c.stats()
        c.timing_enable(True)
        for _ in range(reps):
            event()
        tm = c.timing()
        c.timing_enable(False)
        st1 = c.stats()
    finally:
        c.close()
    n_u = (st1["unique_experts"] - st0["unique_experts"]) / reps
    rows = T * k
    f1 = 2.0 * rows * (2 * w.inter) * w.hidden     # gate/up: [rows x H] . [H x 2I]
    f2 = 2.0 * rows * w.hidden * w.inter           # down: [rows x I] . [I x H]
    g1 = tm["gemm1_ms"] / max(1, tm["gemm1_n"])
    g2 = tm["gemm2_ms"] / max(1, tm["gemm2_n"])
    ffn = tm["ffn_ms"] / max(1, tm["ffn_n"])
    both = (f1 + f2) / ((g1 + g2) / 1e3) / 1e12
    return {"kernel": "tc_gemm_kernel (tcgen05.mma kind::f16, TMA tiles): gate/up + SwiGLU, then down"
                      + (" (fp8 weights and their block scales dequantised to fp16 in shared memory; fp16 operands)" if w.wdtype == synth.W_FP8 else ""),
            "workload": f"{w.name}: {T} tokens, hidden {w.hidden}, inter {w.inter}, {E} experts, top-{k}",
            "bound": "tensor", "unit": "TFLOP/s", "peak": peak_tflops, "launches": tm["gemm1_n"],
            "gateup_ms": g1, "down_ms": g2, "ffn_ms": ffn, "unique_experts": n_u,
            "gateup_tflops": f1 / (g1 / 1e3) / 1e12, "down_tflops": f2 / (g2 / 1e3) / 1e12,
            "achieved": both, "frac": both / peak_tflops,
            "ffn_tflops": (f1 + f2) / (ffn / 1e3) / 1e12,
            "misses": st1["misses"] - st0["misses"],
            "flop_per_layer": f1 + f2,
            "how": f"one-layer cache, the same {T}-token chunk every event (all hits after the first); "
                   "CUDA events around each GEMM launch on the compute stream"}


# The prefill chunk at the DeepSeek-V4-Flash-shaped layer dimensions with fp8 block-scaled experts (no
# configured workload prefills this shape: the chunk size is the 35B prefill's).
FP8_PREFILL = W.DSV4_DECODE.replace(name="dsv4flash-shape-prefill-16k-fp8", tokens=16384, steps=1,
                                    routing=W.ROUTE_ZIPF_IID, resize_step=-1, bank_blobs=0)


def ffn_only(w, dev, peak, layers=16, steps=32):
    """The decode FFN kernel with every expert a hit, through the public API:
    a cache of `layers` layers (2 x layers x k slots) whose routing picks the
    same k experts of each layer every step, so after two warm-up steps no
    fetch runs.  The layers' experts are distinct slots (layers x k x
    expert_bytes, larger than L2), so each FFN streams its 8 experts from HBM.
    Two timings: (1) step graphs without event nodes, CUDA events around
    `steps` back-to-back launches: per-layer time in the pipeline, with
    consecutive FFN kernels overlapping launch and set-up (programmatic
    dependent launch); (2) a graph with event nodes around every FFN launch:
    the kernel's own duration."""
    import torch

    from expert_cache_host_layer_gb300.pipeline import ExpertCache, StepGraph, pinned_bank
    k, E = w.top_k, w.num_experts
    if layers * k > E * layers or w.tokens > 8:
        return None
    n_blobs = min(w.blobs, layers * k)
    bank = pinned_bank(n_blobs * w.expert_bytes)
    synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, np.arange(n_blobs), out_ptr=bank.data_ptr())
    act = torch.float32 if w.wdtype == synth.W_F32 else torch.bfloat16
    c = ExpertCache(layers, E, k, w.hidden, w.inter, w.wdtype, 2 * layers * k, 1, bank, n_blobs, fetch_mode=1,
                    device=dev)
    lg = [torch.full((1, E), -1.0, dtype=torch.float32, device=dev) for _ in range(layers)]
    for l in range(layers):
        e0 = (l * k) % (E - k + 1)
        lg[l][0, e0:e0 + k] = torch.arange(k, 0, -1, device=dev, dtype=torch.float32)
    xs = [torch.from_numpy(W.hidden_states(w, 0, l)[:1]).to(dev, act) for l in range(layers)]
    ys = [torch.empty((1, w.hidden), dtype=torch.float32, device=dev) for _ in range(layers)]
    g = StepGraph(c, lg, xs, ys, True)
    gt = StepGraph(c, lg, xs, ys, True, timing=True)
    try:
        for _ in range(2):  # fill, then one all-hit step
            g.launch()
        c.synchronize()
        st0 = c.stats()
        s = c.stream
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            g.launch()
        e1.record(s)
        c.synchronize()
        step_ms = e0.elapsed_time(e1) / steps
        win = []
        for _ in range(8):
            gt.launch()
            win.append(np.asarray(gt.timing()[2]))
        st1 = c.stats()
    finally:
        g.close()
        gt.close()
        c.close()
    us = 1e3 * step_ms / layers
    kus = 1e3 * float(np.mean(win))
    moved = k * w.expert_bytes
    return {"kernel": "ffn_fused_kernel with no fetch (all hits)", "layers": layers, "steps": steps,
            "launch_us": us, "kernel_window_us": kus, "traffic": FFN_ONLY_TRAFFIC_PER_LAUNCH.get(w.name),
            "bytes_per_launch": moved, "achieved": moved / (us / 1e6) / 1e9, "peak": peak,
            "frac": moved / (us / 1e6) / 1e9 / peak, "unit": "GB/s",
            "achieved_window": moved / (kus / 1e6) / 1e9, "frac_window": moved / (kus / 1e6) / 1e9 / peak,
            "misses": st1["misses"] - st0["misses"],
            "how": "launch_us: CUDA events around back-to-back launches of a 16-layer all-hit step graph, per "
                   "layer (route kernels run ahead on their own stream); kernel_window_us: event nodes around "
                   "each FFN launch in a timing graph"}


def bank_warm(w, dev, bank, n_blobs):
    """Reads every blob of the bank once from the GPU over the host link,
    through the library's own miss path (a throwaway 2E-slot cache routes E/k
    tokens per layer so that every expert of the layer misses), before
    anything is timed: a serving process has long since touched its whole
    bank, while the first GPU reads of freshly written host memory were
    measured at a fraction of the link's rate on some boxes.  Returns
    seconds."""
    import torch

    from expert_cache_host_layer_gb300.pipeline import ExpertCache
    t0 = time.perf_counter()
    E, k = w.num_experts, w.top_k
    T = (E + k - 1) // k
    lg = torch.full((T, E), -1.0, dtype=torch.float32)
    for e in range(E):
        lg[e // k, e] = 1.0
    lg = lg.to(dev)
    x = torch.zeros((T, w.hidden), dtype=torch.float32 if w.wdtype == synth.W_F32 else torch.bfloat16, device=dev)
    y = torch.empty((T, w.hidden), dtype=torch.float32, device=dev)
    c = ExpertCache(w.num_layers, E, k, w.hidden, w.inter, w.wdtype, 2 * E, T, bank, n_blobs, fetch_mode=1,
                    device=dev)
    try:
        for layer in range(min(w.num_layers, (n_blobs + E - 1) // E)):
            c.route_classify(layer, lg)
            c.fetch_misses(layer)
            c.moe_forward(layer, x, y)
        c.synchronize()
    finally:
        c.close()
    return time.perf_counter() - t0


def link_ceilings(w, dev, bank, n_blobs):
    """Host-link ceilings measured on this machine, outside the timed region:
    the copy engine (one cudaMemcpyAsync per blob, as the copy-engine fetch
    does; best of 3 rounds of 32 blobs) and the SM-pull fetch kernel alone
    (a fresh cache routes 32 i.i.d. tokens at one layer: ~100 misses, all
    pulled by one kernel) at 8 layers spread over the bank."""
    import torch

    import synth as S
    from expert_cache_host_layer_gb300.pipeline import ExpertCache
    eb = w.expert_bytes
    n = 32
    d = torch.empty(n * eb, dtype=torch.uint8, device=dev)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    best_ce = 0.0
    for _ in range(3):
        s0.record()
        for i in range(n):
            d[i * eb:(i + 1) * eb].copy_(bank[i * eb:(i + 1) * eb], non_blocking=True)
        s1.record()
        torch.cuda.synchronize(dev)
        best_ce = max(best_ce, n * eb / (s0.elapsed_time(s1) / 1e3) / 1e9)
    del d
    pulls = []
    for l in np.linspace(0, w.num_layers - 1, 8).astype(int).tolist():
        c = ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, 1024, 32, bank,
                        n_blobs, fetch_mode=1, device=dev)
        try:
            lg = torch.from_numpy(S.router_iid(7, 0, l, 32, w.num_experts)).to(dev)
            st0 = c.stats()              # the route kernel counts the misses' bytes
            c.route_classify(l, lg)
            c.synchronize()
            c.timing_enable(True)
            c.fetch_misses(l)
            c.synchronize()
            tm = c.timing()
            st1 = c.stats()
            pulls.append((st1["bytes_fetched"] - st0["bytes_fetched"]) / (tm["fetch_ms"] / 1e3) / 1e9)
        finally:
            c.close()
    return {"copy_engine_gbs": best_ce, "sm_pull_gbs": float(np.mean(pulls)), "sm_pull_max_gbs": float(max(pulls)),
            "sm_pull_per_layer_gbs": [round(v, 1) for v in pulls],
            "how": "copy engine: best of 3 x 32 one-blob cudaMemcpyAsync H2D from the pinned bank; SM pull: "
                   "pull_misses_kernel alone, ~100 missed blobs of one layer per launch, 8 layers across the bank"}


class DecodeBench:
    """One decode workload through captured step graphs on one cache: the
    cache is first filled to steady state by `fill` untimed steps of the same
    routing stream (the miss rate of the first steps is compulsory misses of a
    cold cache, not the workload's), then `warmup` untimed steps, then the
    timed passes.  Step s of the routing/hidden-state stream is used once."""

    def __init__(self, w, dev, bank, n_blobs, args, steps_needed, rank=0):
        import torch

        from expert_cache_host_layer_gb300.pipeline import ExpertCache, StepGraph
        self.w, self.dev, self.args = w, dev, args
        self.L, self.T = w.num_layers, w.tokens
        wl = w.replace(steps=steps_needed, seed=w.seed + rank)  # independent replicas per rank
        self.logits_h = W.router_logits(wl)  # [S][L][T][E]
        self.x_h = np.stack([np.stack([W.hidden_states(wl, s, l) for l in range(self.L)])
                             for s in range(steps_needed)])
        self.act = torch.float32 if w.wdtype == synth.W_F32 else torch.bfloat16
        self.logits_d = torch.from_numpy(self.logits_h).to(dev)
        self.x_d = torch.from_numpy(self.x_h).to(dev, self.act)
        self.lg_buf = torch.empty_like(self.logits_d[0])
        self.x_buf = torch.empty_like(self.x_d[0])
        self.y_buf = torch.empty((self.L, self.T, w.hidden), dtype=torch.float32, device=dev)
        self.double = not args.serial
        self.cache = ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, w.num_slots,
                                 self.T, bank, n_blobs, fetch_mode=args.fetch_mode, pull_ctas=args.pull_ctas,
                                 copy_streams=args.copy_streams, fetch_warps=args.fetch_warps, device=dev)
        self.stream = self.cache.stream
        self.StepGraph = StepGraph
        self.graphs = self._graphs(False)
        self.next = 0  # next step of the stream
        self.last_launches = None  # (n_unique, blobs copied, window ms) per FFN launch of the last timing pass

    def _graphs(self, timing):
        return [self.StepGraph(self.cache, list(self.lg_buf), list(self.x_buf), list(self.y_buf), self.double,
                               timing=timing) for _ in range(2)]

    def regraph(self):
        """After a resize the slot pool may have moved: capture the graphs again."""
        for g in self.graphs:
            g.close()
        self.graphs = self._graphs(False)

    def step(self, gs, i):
        s = self.next
        self.lg_buf.copy_(self.logits_d[s], non_blocking=True)
        self.x_buf.copy_(self.x_d[s], non_blocking=True)
        gs[i % 2].launch()
        self.next += 1

    def run(self, n):
        for i in range(n):
            self.step(self.graphs, i)
        self.cache.synchronize()

    def timed(self, n, world=1, sampler=None):
        """n steps timed with CUDA events on the compute stream, barrier and
        synchronize on both sides; returns (ms, stats delta)."""
        import torch
        self.cache.synchronize()
        st0 = self.cache.stats()
        if sampler:
            sampler.start()
        barrier(world)
        torch.cuda.synchronize(self.dev)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(self.stream)
        for i in range(n):
            self.step(self.graphs, i)
        ev1.record(self.stream)
        self.cache.synchronize()
        torch.cuda.synchronize(self.dev)
        barrier(world)
        clocks = sampler.stop() if sampler else None
        st1 = self.cache.stats()
        return ev0.elapsed_time(ev1), {k: st1[k] - st0[k] for k in st1}, clocks

    def e2e(self, n, world=1):
        """n steps end to end through the C ABI: each step copies its logits and
        hidden states from pinned host memory, runs, and copies y back to
        pinned host memory; wall clock around the whole."""
        import torch
        s0 = self.next
        lg_pin = torch.from_numpy(self.logits_h[s0:s0 + n]).pin_memory()
        x_pin = torch.from_numpy(self.x_h[s0:s0 + n]).to(self.act).pin_memory()
        y_pin = torch.empty((n, self.L, self.T, self.w.hidden), dtype=torch.float32).pin_memory()
        self.cache.synchronize()
        barrier(world)
        torch.cuda.synchronize(self.dev)
        t0 = time.perf_counter()
        for i in range(n):
            self.lg_buf.copy_(lg_pin[i], non_blocking=True)
            self.x_buf.copy_(x_pin[i], non_blocking=True)
            self.graphs[i % 2].launch()
            y_pin[i].copy_(self.y_buf, non_blocking=True)
        self.cache.synchronize()
        torch.cuda.synchronize(self.dev)
        dt = max_over_ranks(time.perf_counter() - t0, world)
        self.next += n
        return {"value": world * n * self.T / dt, "unit": "tokens/s", "ms_per_step": 1e3 * dt / n,
                "h2d_bytes_per_step": int(lg_pin[0].numel() * 4 + x_pin[0].numel() * x_pin.element_size()),
                "d2h_bytes_per_step": int(self.y_buf.numel() * 4)}

    def timing_pass(self, n):
        """n steps through graphs with event nodes around every route, fetch and
        FFN launch, plus each layer's plan read back after the step.  Per
        layer l the FFN window w_l is the fused kernel's duration (it also
        copies layer l+1's misses over the host link); layer 0's misses are
        copied by a pull kernel at the step's start."""
        tg = self._graphs(True)
        L, eb = self.L, self.w.expert_bytes
        ffn, route, fetch0, nmiss, nuniq, step_ms = [], [], [], [], [], []
        try:
            for i in range(n):
                self.step(tg, i)
                r, fe, f, st_ms = tg[i % 2].timing()
                plans = [self.cache.plan(l) for l in range(L)]
                ffn.append(np.asarray(f))
                route.append(np.asarray(r))
                fetch0.append(float(fe[0]))
                nmiss.append(np.array([len(p["miss_expert"]) for p in plans]))
                nuniq.append(np.array([len(p["unique"]) for p in plans]))
                step_ms.append(st_ms)
        finally:
            for g in tg:
                g.close()
        ffn, route, nmiss, nuniq = np.stack(ffn), np.stack(route), np.stack(nmiss), np.stack(nuniq)
        carried = np.zeros_like(nmiss)
        carried[:, :-1] = nmiss[:, 1:]   # FFN(l) copies layer l+1's misses
        marginal = marginal_link(carried, ffn, eb)
        # the FFN alone, in the pipeline: the fit's intercept (at batch 4/8
        # nearly every launch copies something, and the few that copy nothing
        # are not typical), else the median window of the launches that copied
        # nothing
        plain = ffn[carried == 0]
        if marginal and marginal["intercept_us"] > 0:
            f_alone = marginal["intercept_us"] / 1e3
        else:
            f_alone = float(np.median(plain)) if plain.size else float(np.median(ffn))
        exposed = np.clip(ffn - f_alone, 0.0, None).sum(axis=1) + np.asarray(fetch0)
        # host link: bytes over the windows that moved them
        link_bytes = float(nmiss.sum()) * eb
        link_ms = float(ffn[carried > 0].sum() + np.asarray(fetch0)[nmiss[:, 0] > 0].sum())
        hbm_bytes = (nuniq + carried) * eb   # per FFN launch: expert reads + copied blobs written
        self.last_launches = (nuniq.ravel().astype(np.float64), carried.ravel().astype(np.float64),
                              ffn.ravel().astype(np.float64))
        return {"steps": n, "ffn_us_per_launch": 1e3 * float(ffn.mean()),
                "ffn_us_alone_in_pipeline": 1e3 * f_alone,
                "ffn_ms_per_step": float(ffn.sum(axis=1).mean()),
                "route_us_per_launch": 1e3 * float(route.mean()),
                "step_ms_with_event_nodes": float(np.mean(step_ms)),
                "gaps_ms_per_step": float(np.mean(step_ms) - ffn.sum(axis=1).mean() - np.mean(fetch0)),
                "exposed_copy_ms_per_step": float(exposed.mean()),
                "link_gbs": link_bytes / (link_ms / 1e3) / 1e9 if link_ms > 0 else None,
                "link_marginal": marginal,
                "miss_bytes_per_step": link_bytes / n,
                "ffn_hbm_bytes_per_launch": float(hbm_bytes.mean()),
                "ffn_read_bytes_per_launch": float((nuniq * eb).mean()),
                "note": "route runs on its own stream ahead of the FFNs (off the critical path); the FFN "
                        "windows are serial on the compute stream: step = layer-0 pull + FFN windows + gaps; "
                        "ffn_us_alone_in_pipeline = the intercept of link_marginal's fit (the window of an FFN "
                        "that copies nothing, event nodes included); exposed copy = the windows beyond it + "
                        "the layer-0 pull"}

    def close(self):
        for g in self.graphs:
            g.close()
        self.cache.close()


def marginal_link(carried, window_ms, eb):
    """The marginal host-link rate in the pipeline: each FFN window (ms)
    against the number of blobs its kernel copied, least squares; the slope
    is the link time one more blob costs, the intercept the window of an FFN
    that copies nothing (event nodes included).  None without two distinct
    copy counts."""
    xs = np.asarray(carried, dtype=np.float64).ravel()
    ys = np.asarray(window_ms, dtype=np.float64).ravel()
    if np.unique(xs).size < 2:
        return None
    (b0, b1), *_ = np.linalg.lstsq(np.stack([np.ones_like(xs), xs], 1), ys, rcond=None)
    return {"us_per_blob": 1e3 * float(b1), "intercept_us": 1e3 * float(b0),
            "gbs": eb / (float(b1) / 1e3) / 1e9 if b1 > 0 else None,
            "launches_by_blobs_copied": {int(c): int((xs == c).sum()) for c in np.unique(xs)}}


def bound_of_launches(launches, eb, hbm_gbs, link_gbs):
    """Each FFN launch's lower bound: its expert reads at the HBM peak or the
    blobs it copies at the host link's ceiling, whichever takes longer; the
    mean bound against the mean measured window (event nodes included)."""
    if launches is None or not link_gbs:
        return None
    nuniq, carried, ffn_ms = launches
    bound_us = np.maximum(nuniq * eb / (hbm_gbs * 1e3), carried * eb / (link_gbs * 1e3))
    link_bound = carried * eb / (link_gbs * 1e3) > nuniq * eb / (hbm_gbs * 1e3)
    return {"bound_us_per_launch": float(bound_us.mean()), "measured_us_per_launch": float(1e3 * ffn_ms.mean()),
            "frac": float(bound_us.mean() / (1e3 * ffn_ms.mean())), "link_bound_launches": float(link_bound.mean()),
            "hbm_gbs": hbm_gbs, "link_gbs": link_gbs,
            "how": "per launch max(n_unique x expert_bytes / HBM peak, blobs copied x expert_bytes / SM-pull "
                   "ceiling measured alone); frac = mean bound / mean window of the timing pass"}


def decode_block(w, dev, bank, n_blobs, args, steps, warmup, fill, timing_steps, peak, resize=None, link_gbs=None):
    """A compact decode measurement of workload w (its own cache): fill,
    warm-up, `steps` timed, then a timing pass.  `resize` = (slots, fill2):
    after the first timed pass, resize the cache at a safe point, refill for
    fill2 steps and time again."""
    need = fill + warmup + steps + timing_steps + (resize[1] + warmup + steps if resize else 0)
    b = DecodeBench(w, dev, bank, n_blobs, args, need)
    try:
        b.run(fill + warmup)
        ms, d, _ = b.timed(steps)
        tp = b.timing_pass(timing_steps)
        out = {"workload": w.name, "tokens": w.tokens, "slots": w.num_slots, "steps": steps, "warmup": warmup,
               "fill_steps": fill, "tokens_per_s": steps * w.tokens / (ms / 1e3), "ms_per_step": ms / steps,
               "miss_rate": d["misses"] / max(1, d["unique_experts"]),
               "roofline_ffn": {"bound": "hbm", "unit": "GB/s", "peak": peak,
                                "achieved": tp["ffn_read_bytes_per_launch"] / (tp["ffn_us_per_launch"] / 1e6) / 1e9,
                                "achieved_alone_in_pipeline":
                                    tp["ffn_read_bytes_per_launch"] / (tp["ffn_us_alone_in_pipeline"] / 1e6) / 1e9},
               "timing": tp}
        r = out["roofline_ffn"]
        r["frac"] = r["achieved"] / peak
        r["frac_alone_in_pipeline"] = r["achieved_alone_in_pipeline"] / peak
        r["hbm_or_link_bound"] = bound_of_launches(b.last_launches, w.expert_bytes, peak, link_gbs)
        if resize:
            slots, fill2 = resize
            b.cache.synchronize()
            t0 = time.perf_counter()
            b.cache.resize(slots)
            resize_ms = 1e3 * (time.perf_counter() - t0)
            b.regraph()
            b.run(fill2 + warmup)
            ms2, d2, _ = b.timed(steps)
            out["after_resize"] = {"slots": slots, "resize_ms": resize_ms, "fill_steps": fill2,
                                   "tokens_per_s": steps * w.tokens / (ms2 / 1e3), "ms_per_step": ms2 / steps,
                                   "miss_rate": d2["misses"] / max(1, d2["unique_experts"])}
        return out
    finally:
        b.close()


FILL_STEPS = 64  # steady state: the miss rate of the decode stream is counted from step 64 on


def run_ours(args, w):
    import torch

    rank, local, world = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from expert_cache_host_layer_gb300.pipeline import pinned_bank

    if args.slots:
        w = w.replace(num_slots=args.slots)
    n_blobs = args.bank_blobs or w.blobs
    t_setup = time.perf_counter()
    bank = pinned_bank(n_blobs * w.expert_bytes)
    synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, np.arange(n_blobs), out_ptr=bank.data_ptr())
    gen_s = time.perf_counter() - t_setup
    warm_s = bank_warm(w, dev, bank, n_blobs)
    peak, peak_kind = measured_peaks()
    K, Wm = args.steps, args.warmup
    L, T = w.num_layers, w.tokens
    fill = FILL_STEPS

    b = DecodeBench(w, dev, bank, n_blobs, args, fill + Wm + 3 * K + args.timing_steps, rank)
    b.run(fill + Wm)
    # the timed steps (the line's value), then e2e, then the same timed pass again
    sampler = ClockSampler(local)
    ms1, d, clocks = b.timed(K, world, sampler)
    e2e = None if args.no_e2e else b.e2e(K, world)
    ms2, _, _ = b.timed(K, world)
    tp = b.timing_pass(args.timing_steps)
    if args.trace and rank == 0:
        print(json.dumps(tp), file=sys.stderr)
    launches = d["kernel_launches"]
    main_launches = b.last_launches
    b.close()
    elapsed_ms = max_over_ranks(ms1, world)
    tokens = world * K * T
    value = tokens / (elapsed_ms / 1e3)

    ffn_alone = ffn_only(w, dev, peak) if rank == 0 and T <= 8 else None
    link = None
    if rank == 0 and not args.no_link:
        try:
            link = link_ceilings(w, dev, bank, n_blobs)
        except Exception as ex:
            link = {"error": str(ex)[:200]}
    link_pull = (link or {}).get("sm_pull_gbs")
    blocks = {}
    if rank == 0 and not args.no_blocks:
        for wb in (W.QWEN35B_DECODE_B4, W.QWEN35B_DECODE_B8):
            blocks[wb.name] = decode_block(wb, dev, bank, n_blobs, args, max(8, K // 2), 3, fill, 16, peak,
                                           link_gbs=link_pull)
        blocks["prefill"] = prefill_measure(dev, measured_bf16_tflops())
        blocks["prefill"]["gemm_alone"] = prefill_gemm_only(dev, measured_bf16_tflops())
        blocks["prefill"]["gemm_alone_fp8"] = prefill_gemm_only(dev, measured_bf16_tflops(), w=FP8_PREFILL)
        wd = W.DSV4_DECODE
        dbank = pinned_bank(wd.blobs * wd.expert_bytes)
        synth.expert_blobs(wd.seed, wd.hidden, wd.inter, wd.wdtype, np.arange(wd.blobs), out_ptr=dbank.data_ptr())
        bank_warm(wd, dev, dbank, wd.blobs)
        blocks[wd.name] = decode_block(wd, dev, dbank, wd.blobs, args, max(8, K // 2), 3, 40, 8, peak,
                                       resize=(wd.resize_slots, 24), link_gbs=link_pull)
        blocks[wd.name]["bank"] = f"aliased: {wd.blobs} physical blobs of {wd.expert_bytes} B for " \
                                  f"{wd.keys} (layer, expert) keys"
        del dbank
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline(w, args.cpu_baseline_steps)
        except Exception as ex:  # reported, not fatal
            cpu = {"value": None, "unit": "tokens/s", "cores": cpu_workers(), "kind": "oracle",
                   "sample": f"failed: {ex}"[:300]}

    if rank == 0:
        eb = w.expert_bytes
        bytes_launch = tp["ffn_hbm_bytes_per_launch"]
        achieved = bytes_launch / (tp["ffn_us_per_launch"] / 1e6) / 1e9
        link_ceiling = (link or {}).get("sm_pull_gbs") or None
        need_ms = tp["miss_bytes_per_step"] / (link_ceiling * 1e9) * 1e3 if link_ceiling else None
        ffn_ms = L * ffn_alone["launch_us"] / 1e3 if ffn_alone else None
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": Wm, "ms_per_step": elapsed_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.wdtype == synth.W_BF16 else
            ("f32" if w.wdtype == synth.W_F32 else "fp8e4m3"), "data": "synthetic",
            "config": dict(workload_config(w, world, n_blobs), fetch_mode=["copy_engine", "sm_pull"][args.fetch_mode],
                           double_buffer=not args.serial, step_graph=True, cache_fill_steps=fill,
                           cache_fill="the routing stream's first 64 steps run untimed before the warm-up, so "
                                      "the timed steps see the steady-state miss rate, not a cold cache's",
                           bank_warm="every blob of the host bank is read once from the GPU through the "
                                     "library's miss path before the fill (setup_s.bank_warm), as a serving "
                                     "process has long since done; the timed steps still copy every miss"),
            "miss_rate": d["misses"] / max(1, d["unique_experts"]),
            "repeat_ms_per_step": [ms1 / K, ms2 / K],
            "expert_gemm_gbs": achieved,
            "exposed_copy_ms_per_step": tp["exposed_copy_ms_per_step"],
            "miss_copy": {"gbs": tp["link_gbs"], "gbs_marginal": (tp["link_marginal"] or {}).get("gbs"),
                          "bytes_per_step": d["bytes_fetched"] / K,
                          "mode": ["copy_engine", "sm_pull"][args.fetch_mode], "link": link,
                          "link_time_needed_ms": need_ms, "ffn_time_ms": ffn_ms,
                          "fits_link_budget": (need_ms <= ffn_ms) if need_ms and ffn_ms else None,
                          "how": "gbs = miss bytes of the timing pass / the durations of the kernels that "
                                 "copied them (each fused FFN copies the next layer's misses; layer 0's come "
                                 "from a pull kernel; a window also holds the FFN's own start and the event "
                                 "nodes); gbs_marginal = expert bytes / the extra window one more copied blob "
                                 "costs (least squares over the timing pass's FFN launches); fits_link_budget: "
                                 "miss bytes / sm_pull ceiling <= L x FFN-alone time"},
            "per_kernel": tp,
            "roofline": {"kernel": "ffn_fused_kernel: one launch per layer (gate/up, SwiGLU, down, combine; "
                                   "a programmatic dependent of the previous layer's) that also copies the "
                                   "next layer's misses; CUDA event nodes around each launch in the timing "
                                   "pass",
                         "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "traffic": pipeline_traffic(w.name, tp["ffn_read_bytes_per_launch"] / w.expert_bytes),
                         "traffic_how": "DRAM bytes per unique expert read x the mean unique experts + the "
                                        "writes per launch, from an ncu capture of a small case of this kernel "
                                        "(the copied blobs' writes reach DRAM after the launch, from L2)",
                         "bytes_per_launch": bytes_launch,
                         "bytes_def": "n_unique x expert_bytes read + n_miss(next layer) x expert_bytes written",
                         "launch_us": tp["ffn_us_per_launch"], "ffn_only": ffn_alone,
                         "hbm_or_link_bound": bound_of_launches(main_launches, w.expert_bytes, peak, link_pull)},
            "cpu_baseline": cpu,
            "blocks": blocks,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
            "setup_s": {"bank_generate": round(gen_s, 1), "bank_warm": round(warm_s, 2)},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    w = W.ALL[args.workload]
    if args.ffn_only:
        import torch
        print(json.dumps(ffn_only(w, torch.device("cuda", 0), measured_peaks()[0])), flush=True)
        return
    if args.prefill_gemm_only:
        import torch
        pw = FP8_PREFILL if w.wdtype == synth.W_FP8 else W.QWEN35B_PREFILL
        if args.gemm_experts:
            pw = pw.replace(num_experts=args.gemm_experts)
        if args.gemm_tokens:
            pw = pw.replace(tokens=args.gemm_tokens)
        print(json.dumps(prefill_gemm_only(torch.device("cuda", 0), measured_bf16_tflops(), w=pw)), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
