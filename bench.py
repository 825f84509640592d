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
    p.add_argument("--steps", type=int, default=496)
    p.add_argument("--warmup", type=int, default=16)
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
    p.add_argument("--prefill", action="store_true",
                   help="also measure the 16,384-token prefill chunk (40 layers) and report it under 'prefill'")
    p.add_argument("--trace", action="store_true", help="print one step's per-layer timeline to stderr")
    p.add_argument("--prefill-gemm-only", action="store_true",
                   help="only time the prefill chunk's two tensor-core GEMMs (all hits, no fetch) and print them")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--timing-steps", type=int, default=64,
                   help="steps of the second timed pass (graphs with per-phase events) for the roofline")
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

def oracle_sample(w: W.Workload, seconds: float, logits=None):
    """Time the CPU oracle (routing, LRU simulation, fp64 FFN) on consecutive
    steps of workload w until `seconds` of oracle time have passed (at least
    one step).  Input generation (the expert blobs, hidden states) is not
    timed.  The cache simulation starts cold at step 0.  Returns (tokens/s,
    steps, oracle seconds)."""
    from oracle import ffn as offn
    from oracle import routing as orouting
    from oracle.cache import ExpertCacheOracle
    if logits is None:
        logits = W.router_logits(w.replace(steps=min(w.steps, 64)))
    ref = ExpertCacheOracle(w.num_layers, w.num_experts, w.num_slots)
    spent = 0.0
    steps = 0
    while steps < logits.shape[0]:
        for l in range(w.num_layers):
            topk = orouting.topk(logits[steps, l], w.top_k)
            raw = {e: synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, [w.blob_of(l, e)])
                   for e in sorted({int(v) for v in topk.ravel()})}
            x = W.hidden_states(w, steps, l)
            t0 = time.perf_counter()
            idx, gw = orouting.route(logits[steps, l], w.top_k)
            ref.event(l, idx)
            blobs = {e: offn.dequant_blob(b, w.hidden, w.inter, w.wdtype) for e, b in raw.items()}
            offn.moe_ffn(x, idx, gw, lambda e: blobs[e])
            spent += time.perf_counter() - t0
        steps += 1
        if spent >= seconds:
            break
    return steps * w.tokens / spent, steps, spent


def cpu_baseline_subprocess(w: W.Workload, seconds: float):
    """Run the oracle sample in a child process pinned to one BLAS thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = ("import json,sys; sys.path.insert(0, %r); import bench; from synth import workloads as W; "
            "v, s, dt = bench.oracle_sample(W.ALL[%r], %r); print(json.dumps([v, s, dt]))") % (ROOT, w.name, seconds)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        raise RuntimeError("oracle baseline failed: " + r.stderr[-2000:])
    v, s, dt = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"first {s} decode steps x {w.num_layers} layers of {w.name} (routing, LRU simulation, "
                      f"fp64 SwiGLU FFN), {dt:.1f} s on 1 host thread"}


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
    # each step: the oracle over a bounded sample of steps of the same workload
    per = []
    total_steps = 0
    seconds = max(1.0, min(args.cpu_seconds, 20.0) / max(1, args.steps))
    logits = W.router_logits(w.replace(steps=min(w.steps, 64)))
    for i in range(args.warmup + args.steps):
        v, s, dt = oracle_sample(w, seconds, logits)
        if i >= args.warmup:
            per.append(dt / max(1, s))
            total_steps += s
    ms = 1e3 * statistics.mean(per)
    value = w.tokens / (ms / 1e3)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.gpus, args.bank_blobs or w.blobs),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{total_steps} decode steps (cold cache start) of {w.name}, "
                                       "single host thread"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- our arm

# dram__bytes_read.sum + dram__bytes_write.sum of one ffn_fused_kernel launch
# (35B-shaped bf16 decode layer, 8 unique experts), mean of the two launches
# of the ncu --set full capture summarised under profiles/.  It belongs to the
# kernel as captured: set it to None whenever that kernel changes.
FFN_TRAFFIC_PER_LAUNCH = {"qwen35b-a3b-shape-decode-b1": ((50.404352 + 0.292096) + (50.404608 + 0.148224)) / 2 * 1e6}


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
    out["note"] = ("step graph with timing event nodes, 40 layers, one 16,384-token chunk each; FFN = grouped "
                   "mma.sync bf16 GEMMs (gate/up + SwiGLU, down) + combine; times from the event nodes")
    return out


def prefill_gemm_only(dev, peak_tflops, reps=6):
    """The prefill chunk's two tensor-core GEMMs alone, through the public
    API: a one-layer cache of 512 slots routes the same 16,384-token chunk
    every event, so after the first event every unique expert hits and no
    fetch runs beside the GEMMs.  The library's event timing brackets the
    gate/up + SwiGLU GEMM and the down GEMM of each forward.  The weights the
    GEMMs stream (~214 experts x 6.3 MB) are larger than L2."""
    import torch

    from expert_cache_host_layer_gb300.pipeline import ExpertCache, pinned_bank
    w = W.QWEN35B_PREFILL
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
    return {"kernel": "tc_gemm_kernel (tcgen05.mma kind::f16, TMA tiles): gate/up + SwiGLU, then down",
            "bound": "tensor", "unit": "TFLOP/s", "peak": peak_tflops, "launches": tm["gemm1_n"],
            "gateup_ms": g1, "down_ms": g2, "ffn_ms": ffn, "unique_experts": n_u,
            "gateup_tflops": f1 / (g1 / 1e3) / 1e12, "down_tflops": f2 / (g2 / 1e3) / 1e12,
            "achieved": both, "frac": both / peak_tflops,
            "ffn_tflops": (f1 + f2) / (ffn / 1e3) / 1e12,
            "misses": st1["misses"] - st0["misses"],
            "flop_per_layer": f1 + f2,
            "how": "one-layer cache, the same 16,384-token chunk every event (all hits after the first); "
                   "CUDA events around each GEMM launch on the compute stream"}


def ffn_only(w, dev, peak):
    """The fused FFN kernel alone, through the public API: a one-layer cache of
    16*k slots whose routing rotates through 16 disjoint sets of k experts, so
    after 16 warm-up events every event hits (no fetch rides along) and each
    FFN streams k experts that the previous 15 events did not touch (16*k
    experts > L2).  Times the kernel with the step graph's event nodes."""
    import torch

    from expert_cache_host_layer_gb300.pipeline import ExpertCache, StepGraph, pinned_bank
    k, E = w.top_k, w.num_experts
    nsets = 16
    n_blobs = nsets * k
    if n_blobs > E:
        return None
    bank = pinned_bank(n_blobs * w.expert_bytes)
    synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, np.arange(n_blobs), out_ptr=bank.data_ptr())
    act = torch.float32 if w.wdtype == synth.W_F32 else torch.bfloat16
    c = ExpertCache(1, E, k, w.hidden, w.inter, w.wdtype, n_blobs, 1, bank, n_blobs, fetch_mode=1, device=dev)
    lg = torch.full((1, E), -1.0, dtype=torch.float32, device=dev)
    x = torch.from_numpy(W.hidden_states(w, 0, 0)[:1]).to(dev, act)
    y = torch.empty((1, w.hidden), dtype=torch.float32, device=dev)
    g = StepGraph(c, [lg], [x], [y], True, timing=True)
    try:
        def launch(j):
            lg.fill_(-1.0)
            lg[0, (j % nsets) * k:(j % nsets + 1) * k] = torch.arange(k, 0, -1, device=dev, dtype=torch.float32)
            g.launch()
        for j in range(2 * nsets):  # fill the slots, then one all-hit round
            launch(j)
        c.synchronize()
        st0 = c.stats()
        ffn_ms = []
        for j in range(64):
            launch(j)
            ffn_ms.append(float(g.timing()[2][0]))
        st1 = c.stats()
    finally:
        g.close()
        c.close()
    us = 1e3 * float(np.mean(ffn_ms))
    moved = k * w.expert_bytes
    return {"kernel": "ffn_fused_kernel with no fetch (all hits)", "launches": len(ffn_ms), "launch_us": us,
            "bytes_per_launch": moved, "achieved": moved / (us / 1e6) / 1e9, "peak": peak,
            "frac": moved / (us / 1e6) / 1e9 / peak, "unit": "GB/s",
            "misses": st1["misses"] - st0["misses"]}


def link_ceilings(cache, w, dev, bank):
    """Host-link ceilings measured on this machine, outside the timed region:
    the copy engine (one cudaMemcpyAsync per blob, as the copy-engine fetch
    does) and the SM-pull fetch kernel alone on a cold cache (T=32 i.i.d.
    tokens: ~100+ misses per layer event)."""
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
    c = ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, 1024, 32, bank,
                    cache.bank_blobs, fetch_mode=1, device=dev)
    best_pull = 0.0
    spread = []  # the same over layers spread across the bank (its far pages)
    try:
        for l in list(range(4)) + [9, 19, 29, 39]:
            if l >= w.num_layers:
                continue
            lg = torch.from_numpy(S.router_iid(7, 0, l, 32, w.num_experts)).to(dev)
            st0 = c.stats()
            c.route_classify(l, lg)
            c.synchronize()
            c.timing_enable(True)
            c.fetch_misses(l)
            c.synchronize()
            tm = c.timing()
            st1 = c.stats()
            c.timing_enable(False)
            gbs = (st1["bytes_fetched"] - st0["bytes_fetched"]) / (tm["fetch_ms"] / 1e3) / 1e9
            if 0 < l < 4:
                best_pull = max(best_pull, gbs)
            elif l >= 4:
                spread.append(gbs)
            c.close()
            c = ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, 1024, 32, bank,
                            cache.bank_blobs, fetch_mode=1, device=dev)
    finally:
        c.close()
    return {"copy_engine_gbs": best_ce, "sm_pull_gbs": best_pull,
            "sm_pull_spread_gbs": float(np.mean(spread)) if spread else None,
            "how": "best of a few isolated runs: 32 x one-blob cudaMemcpyAsync H2D from pinned memory; "
                   "pull_misses_kernel on a cold cache (first layers' blobs; spread: layers across the bank)"}


def run_ours(args, w):
    import torch

    rank, local, world = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from expert_cache_host_layer_gb300.pipeline import ExpertCache, StepGraph, pinned_bank

    if args.slots:
        w = w.replace(num_slots=args.slots)
    n_blobs = args.bank_blobs or w.blobs
    t_setup = time.perf_counter()
    bank = pinned_bank(n_blobs * w.expert_bytes)
    synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, np.arange(n_blobs), out_ptr=bank.data_ptr())
    gen_s = time.perf_counter() - t_setup

    steps_total = args.warmup + args.steps + args.timing_steps
    wl = w.replace(steps=steps_total, seed=w.seed + rank)  # independent replicas per rank
    logits_h = W.router_logits(wl)                             # [S][L][T][E]
    x_h = np.stack([np.stack([W.hidden_states(wl, s, l) for l in range(w.num_layers)]) for s in range(steps_total)])
    act = torch.float32 if w.wdtype == synth.W_F32 else torch.bfloat16
    logits_d = torch.from_numpy(logits_h).to(dev)
    x_d = torch.from_numpy(x_h).to(dev, act)
    L, T = w.num_layers, w.tokens
    # fixed per-layer buffers the captured step reads and writes
    lg_buf = torch.empty_like(logits_d[0])
    x_buf = torch.empty_like(x_d[0])
    y_buf = torch.empty((L, T, w.hidden), dtype=torch.float32, device=dev)
    double = not args.serial

    def make_cache():
        return ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, w.num_slots, T, bank,
                           n_blobs, fetch_mode=args.fetch_mode, pull_ctas=args.pull_ctas,
                           copy_streams=args.copy_streams, fetch_warps=args.fetch_warps, device=dev)

    use_graph = True
    cache = make_cache()
    stream = cache.stream
    # plain graphs for the timed steps; graphs with per-phase event nodes (which
    # slow a step down) only for the second, roofline pass
    graphs = [StepGraph(cache, list(lg_buf), list(x_buf), list(y_buf), double) for _ in range(2)]
    tgraphs = [StepGraph(cache, list(lg_buf), list(x_buf), list(y_buf), double, timing=True) for _ in range(2)]

    def step(s, i, gs):
        lg_buf.copy_(logits_d[s], non_blocking=True)
        x_buf.copy_(x_d[s], non_blocking=True)
        gs[i % 2].launch()

    for s in range(args.warmup):
        step(s, s, graphs)
    cache.synchronize()
    st0 = cache.stats()
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i, s in enumerate(range(args.warmup, args.warmup + args.steps)):
        step(s, i, graphs)
    ev1.record(stream)
    cache.synchronize()
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    elapsed_ms = ev0.elapsed_time(ev1)
    st1 = cache.stats()

    # ---- second timed pass: per-layer route / fetch / FFN event times -----
    acc = {"route": 0.0, "fetch": 0.0, "ffn": 0.0, "n": 0, "step": 0.0}
    if args.fetch_mode == 0:  # copy-engine fetches are timed by the library's copy thread
        cache.timing_enable(True)
    t_first = args.warmup + args.steps
    for i, s in enumerate(range(t_first, t_first + args.timing_steps)):
        step(s, i, tgraphs)
        if i > 0:  # the previous step's events (it is done or nearly so)
            r, fe, f, st_ms = tgraphs[(i - 1) % 2].timing()
            acc["route"] += r.sum(); acc["fetch"] += fe.sum(); acc["ffn"] += f.sum(); acc["n"] += 1
            acc["step"] += st_ms
    cache.synchronize()
    if args.timing_steps:
        r, fe, f, st_ms = tgraphs[(args.timing_steps - 1) % 2].timing()
        acc["route"] += r.sum(); acc["fetch"] += fe.sum(); acc["ffn"] += f.sum(); acc["n"] += 1
        acc["step"] += st_ms
    tm = {"route_ms": acc["route"], "fetch_ms": acc["fetch"], "ffn_ms": acc["ffn"],
          "route_n": acc["n"] * L, "fetch_n": acc["n"] * L, "ffn_n": acc["n"] * L}
    if args.fetch_mode == 0:
        ct = cache.timing()
        tm["fetch_ms"], tm["fetch_n"] = ct["fetch_ms"], ct["fetch_n"]
        cache.timing_enable(False)
    st2 = cache.stats()
    if args.trace and rank == 0 and args.timing_steps:
        tr = tgraphs[(args.timing_steps - 1) % 2].trace()
        print("layer  route_b route_e  fetch_b fetch_e  ffn_b  ffn_e  (us from step start)", file=sys.stderr)
        for l in range(L):
            print(f"{l:5d} " + " ".join(f"{1e3 * v:7.1f}" for v in tr[l]), file=sys.stderr)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    tokens = world * args.steps * T
    value = tokens / (elapsed_ms / 1e3)

    d = {k: st1[k] - st0[k] for k in st1}    # the timed steps
    d2 = {k: st2[k] - st1[k] for k in st1}   # the roofline pass
    eb = w.expert_bytes
    ffn_bytes_per_launch = d2["unique_experts"] * eb / max(1, tm["ffn_n"])
    ffn_ms = tm["ffn_ms"] / max(1, tm["ffn_n"])
    peak, peak_kind = measured_peaks()
    achieved = ffn_bytes_per_launch / (ffn_ms / 1e3) / 1e9 if ffn_ms > 0 else None
    fetch_gbs = d2["bytes_fetched"] / max(1e-9, tm["fetch_ms"] / 1e3) / 1e9 if tm["fetch_ms"] > 0 else None
    n_tsteps = max(1, acc["n"])
    for g in graphs + tgraphs:
        g.close()

    # ---- end to end through the C ABI with host buffers -------------------
    e2e = None
    if not args.no_e2e:
        lg_pin = torch.from_numpy(logits_h[args.warmup:]).pin_memory()
        x_pin = torch.from_numpy(x_h[args.warmup:]).to(act).pin_memory()
        y_pin = torch.empty((args.steps, L, T, w.hidden), dtype=torch.float32).pin_memory()
        cache2 = make_cache()
        g2 = StepGraph(cache2, list(lg_buf), list(x_buf), list(y_buf), double) if use_graph else None
        for s in range(args.warmup):  # same warm state as the device-timed run
            lg_buf.copy_(logits_d[s]); x_buf.copy_(x_d[s])
            g2.launch() if g2 else cache2.run_step(list(lg_buf), list(x_buf), list(y_buf), double_buffer=double)
        cache2.synchronize()
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for i in range(args.steps):
            lg_buf.copy_(lg_pin[i], non_blocking=True)
            x_buf.copy_(x_pin[i], non_blocking=True)
            g2.launch() if g2 else cache2.run_step(list(lg_buf), list(x_buf), list(y_buf), double_buffer=double)
            y_pin[i].copy_(y_buf, non_blocking=True)
        cache2.synchronize()  # polls: the copy thread may still have copies to enqueue
        torch.cuda.synchronize(dev)
        e2e_s = max_over_ranks(time.perf_counter() - t0, world)
        if g2:
            g2.close()
        cache2.close()
        e2e = {"value": world * args.steps * T / e2e_s, "unit": "tokens/s",
               "h2d_bytes_per_step": int(lg_pin[0].numel() * 4 + x_pin[0].numel() * x_pin.element_size()),
               "d2h_bytes_per_step": int(y_buf.numel() * 4)}

    link = None
    if rank == 0 and not args.no_link:
        try:
            link = link_ceilings(cache, w, dev, bank)
        except Exception as ex:
            link = {"error": str(ex)[:200]}
    ffn_alone = None
    if rank == 0 and T <= 8:
        ffn_alone = ffn_only(w, dev, peak)
    prefill = None
    if rank == 0 and args.prefill:
        prefill = prefill_measure(dev, measured_bf16_tflops())

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline_subprocess(w, args.cpu_seconds)
        except Exception as ex:  # reported, not fatal
            cpu = {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": f"failed: {ex}"[:300]}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.wdtype == synth.W_BF16 else
            ("f32" if w.wdtype == synth.W_F32 else "fp8e4m3"), "data": "synthetic",
            "config": dict(workload_config(w, world, n_blobs),
                           fetch_mode=["copy_engine", "sm_pull"][args.fetch_mode], double_buffer=double,
                           step_graph=use_graph),
            "miss_rate": d["misses"] / max(1, d["unique_experts"]),
            "exposed_copy_ms_per_step": (elapsed_ms / args.steps - L * ffn_alone["launch_us"] / 1e3)
            if ffn_alone else None,
            "expert_gemm_gbs": achieved,
            "miss_copy": {"gbs": fetch_gbs, "bytes_per_step": d["bytes_fetched"] / args.steps,
                          "mode": ["copy_engine", "sm_pull"][args.fetch_mode], "link": link},
            "phase_ms_per_step": dict({k: tm[f"{k}_ms"] / n_tsteps for k in ("route", "fetch", "ffn")},
                                      step=acc["step"] / n_tsteps, steps=acc["n"],
                                      note="sums of per-layer kernel times from a second timed pass with "
                                           "timing graphs (event nodes around every phase)"),
            "roofline": {"kernel": "ffn_fused_kernel: one cooperative launch per layer (gate/up, SwiGLU, down, "
                                   "combine), timed by event nodes around it in the timing pass",
                         "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak if achieved else None,
                         "peak_kind": peak_kind, "traffic": FFN_TRAFFIC_PER_LAUNCH.get(w.name),
                         "bytes_per_launch": ffn_bytes_per_launch,
                         "launch_us": ffn_ms * 1e3, "ffn_only": ffn_alone},
            "cpu_baseline": cpu,
            "prefill": prefill,
            "e2e": e2e,
            "gpu_launches": d["kernel_launches"],
            "clocks": clocks,
            "setup_s": {"bank_generate": round(gen_s, 1)},
        }
        print(json.dumps(line), flush=True)
    cache.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    w = W.ALL[args.workload]
    if args.prefill_gemm_only:
        import torch
        print(json.dumps(prefill_gemm_only(torch.device("cuda", 0), measured_bf16_tflops())), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
