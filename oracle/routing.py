"""Router top-k and gate weights (oracle).

The pages state only that the model has 256 routed experts and that the
router selects eight per token ("FreeToken vs vLLM on one RTX 3090", section
"Why the performance differs", FreeToken exploits MoE sparsity).  Readings
taken where they are silent:

* Selection is by logit, descending; equal logits are ordered by the lower
  expert index first.  -0.0 and +0.0 compare equal (float comparison).  NaN
  logits are ordered as -inf.  The output order of the k picks is this order.
* Gates are the softmax restricted to the k selected logits,
  w_j = exp(l_j - m) / sum_{i in top-k} exp(l_i - m), m = the largest selected
  logit.  This equals "softmax over all experts, then renormalise the selected
  k", the convention of the Qwen3-MoE family whose shape the decode workload
  uses.
"""
from __future__ import annotations

import numpy as np


def selection_order(logits: np.ndarray) -> np.ndarray:
    """Per row, all expert indices sorted by (logit descending, index ascending)."""
    x = np.asarray(logits, dtype=np.float64)
    x = np.where(np.isnan(x), -np.inf, x)
    x = x + 0.0                                     # -0.0 -> +0.0
    idx = np.broadcast_to(np.arange(x.shape[-1]), x.shape)
    # lexsort: last key is primary -> primary -logit, secondary index
    return np.lexsort((idx, -x), axis=-1)


def topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Top-k expert indices per token, int32 [T, k], in selection order."""
    return selection_order(logits)[..., :k].astype(np.int32)


def gates(logits: np.ndarray, topk_idx: np.ndarray) -> np.ndarray:
    """Gate weights float64 [T, k]: softmax over the selected logits only."""
    x = np.asarray(logits, dtype=np.float64)
    sel = np.take_along_axis(x, np.asarray(topk_idx, dtype=np.int64), axis=-1)
    m = sel.max(axis=-1, keepdims=True)
    p = np.exp(sel - m)
    return p / p.sum(axis=-1, keepdims=True)


def route(logits: np.ndarray, k: int):
    """(topk_idx int32 [T,k], gates float64 [T,k]) for router logits [T,E]."""
    idx = topk(logits, k)
    return idx, gates(logits, idx)
