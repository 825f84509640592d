"""Oracle FFN checks run in host worker processes (spawned, never forked).

A worker regenerates the layer's expert blobs with the same seeded generator
that filled the host bank (the parity run checks separately that the fetched
slots hold exactly those bank bytes), evaluates the oracle FFN in fp64 and
returns the error of the GPU output.  Imports no GPU code.
"""
from __future__ import annotations

import numpy as np

import synth
from oracle import ffn as offn


def ffn_error_job(w, n_blobs, layer, x, idx, gates, y_gpu):
    """(max |diff| / RMS(ref), RMS(diff) / RMS(ref)) of y_gpu against the oracle."""
    cache = {}

    def weights_of(e):
        if e not in cache:
            blob = synth.expert_blobs(w.seed, w.hidden, w.inter, w.wdtype, [(layer * w.num_experts + e) % n_blobs])
            cache[e] = offn.dequant_blob(blob, w.hidden, w.inter, w.wdtype)
        return cache[e]

    yr = offn.moe_ffn(np.asarray(x, dtype=np.float64), idx, gates, weights_of)
    rms = float(np.sqrt(np.mean(yr ** 2))) or 1.0
    d = np.asarray(y_gpu, dtype=np.float64) - yr
    return float(np.abs(d).max() / rms), float(np.sqrt(np.mean(d ** 2)) / rms)
