"""Workload definitions: shapes, cache sizes and input recipes.

These are the synthetic stand-ins for the pages' workloads.  No public
dataset or trained checkpoint is involved: weights, router logits and hidden
states all come from ``synth``.

* tiny: 2 MoE layers x 16 experts, top-2, hidden 256, intermediate 128, fp32
  weights, pure N(0,1) router logits, 64 decode steps of batch 1, 12 slots.
* qwen35b-decode: Qwen3.6-35B-A3B-shaped layers (40 x 256 experts, top-8,
  hidden 2048, intermediate 512, bf16), Zipf(1.1)-biased routing with 70% of
  each step's top-8 kept from the previous step, batch 1, 512 steps, cache of
  3072 slots (30% of the 10240 (layer, expert) keys).
* qwen35b-decode-b4 / -b8: the same shape with 4 / 8 independent decode
  streams sharing one cache of 1740 slots (17% of the bank).
* qwen35b-prefill: one 16,384-token chunk per layer, i.i.d. Zipf-biased
  routing, cold 3072-slot cache.
* dsv4flash-decode: DeepSeek-V4-Flash-shaped layers (24 x 256 experts, top-8,
  hidden 4096, intermediate 2048, fp8 e4m3 with bf16 128x128 block scales),
  batch 1, 1024 steps, 2383 slots (60 GB) resized to 1191 slots (30 GB)
  before step 512.

``bank_blobs`` < L*E selects the aliased host bank: the (layer, expert) key
maps to physical blob (layer*E + expert) mod bank_blobs.  Transfer sizes and
the key space stay the same; only host RAM shrinks.
"""
from __future__ import annotations

import dataclasses

from . import W_BF16, W_F32, W_FP8, expert_bytes

ROUTE_NORMAL = "normal"          # pure N(0,1)
ROUTE_ZIPF_CORR = "zipf_corr"    # N(0,1) + Zipf bias, 70% kept from the previous step
ROUTE_ZIPF_IID = "zipf_iid"      # N(0,1) + Zipf bias, i.i.d. per token


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_layers: int
    num_experts: int
    top_k: int
    hidden: int
    inter: int
    wdtype: int
    tokens: int            # tokens per layer step (decode streams or prefill chunk)
    steps: int
    num_slots: int
    routing: str
    resize_step: int = -1  # step before which the cache is resized (-1: never)
    resize_slots: int = 0
    bank_blobs: int = 0    # 0: full bank (num_layers * num_experts blobs)
    seed: int = 20261202

    @property
    def expert_bytes(self) -> int:
        return expert_bytes(self.hidden, self.inter, self.wdtype)

    @property
    def keys(self) -> int:
        return self.num_layers * self.num_experts

    @property
    def blobs(self) -> int:
        return self.bank_blobs or self.keys

    def blob_of(self, layer: int, expert: int) -> int:
        return (layer * self.num_experts + expert) % self.blobs

    @property
    def act_bf16(self) -> bool:
        return self.wdtype != W_F32

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


TINY = Workload("tiny-2x16-top2-fp32", 2, 16, 2, 256, 128, W_F32, 1, 64, 12, ROUTE_NORMAL)
QWEN35B_DECODE = Workload("qwen35b-a3b-shape-decode-b1", 40, 256, 8, 2048, 512, W_BF16, 1, 512, 3072,
                          ROUTE_ZIPF_CORR)
QWEN35B_DECODE_B4 = QWEN35B_DECODE.replace(name="qwen35b-a3b-shape-decode-b4", tokens=4, num_slots=1740)
QWEN35B_DECODE_B8 = QWEN35B_DECODE.replace(name="qwen35b-a3b-shape-decode-b8", tokens=8, num_slots=1740)
QWEN35B_PREFILL = QWEN35B_DECODE.replace(name="qwen35b-a3b-shape-prefill-16k", tokens=16384, steps=1,
                                         routing=ROUTE_ZIPF_IID)
_DSV4_EB = expert_bytes(4096, 2048, W_FP8)
DSV4_DECODE = Workload("dsv4flash-shape-decode-b1-fp8", 24, 256, 8, 4096, 2048, W_FP8, 1, 1024,
                       int(60e9 // _DSV4_EB), ROUTE_ZIPF_CORR, resize_step=512,
                       resize_slots=int(30e9 // _DSV4_EB), bank_blobs=1024)

ALL = {w.name: w for w in (TINY, QWEN35B_DECODE, QWEN35B_DECODE_B4, QWEN35B_DECODE_B8, QWEN35B_PREFILL,
                           DSV4_DECODE)}


def router_logits(w: Workload):
    """All router logits of a workload: float32 [steps][L][tokens][E].

    Decode workloads draw one routing stream per token (independent streams);
    the prefill workload draws i.i.d. logits per token for its single chunk.
    """
    import numpy as np

    from . import router_decode, router_iid
    if w.routing == ROUTE_ZIPF_IID:
        out = np.empty((w.steps, w.num_layers, w.tokens, w.num_experts), dtype=np.float32)
        for s in range(w.steps):
            for l in range(w.num_layers):
                out[s, l] = router_iid(w.seed, s, l, w.tokens, w.num_experts, 1.1)
        return out
    zipf, keep = (1.1, 0.7) if w.routing == ROUTE_ZIPF_CORR else (0.0, -1.0)
    per_stream = [router_decode(w.seed, b, w.num_layers, w.num_experts, w.top_k, w.steps, zipf, keep)
                  for b in range(w.tokens)]
    return np.ascontiguousarray(np.stack(per_stream, axis=2))


def hidden_states(w: Workload, step: int, layer: int):
    """Hidden states entering the MoE FFN at (step, layer): float32 [tokens][H]
    (bf16-exact values for the bf16 and fp8 workloads)."""
    from . import hidden
    return hidden(w.seed, 0, step, layer, w.tokens, w.hidden, w.act_bf16)
