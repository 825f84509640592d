"""CPU oracle for the per-MoE-layer step of a two-tier expert-offload engine.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it.  It shares no code with the CUDA library
(``expert_cache_host_layer_gb300``); the only common module is ``synth``, which
makes seeded inputs and holds none of the method's arithmetic.

What it computes, each part written as the plain definition, slowly and in
fp64 where floating point is involved:

* ``routing``  - top-k selection and gate weights per token;
* ``cache``    - the global (layer, expert)-keyed slot cache with LRU
                 replacement: dedup, hit classification, victim selection,
                 table updates, and the safe-point resize;
* ``fp8``      - OCP FP8 E4M3 decoding;
* ``ffn``      - expert-blob dequantisation and the SwiGLU expert FFN with the
                 gate-weighted combine;
* ``stream``   - the decision stream of a whole workload (events in step,
                 then layer order, with the safe-point resize);
* ``policies`` - the static placements the pages compare the cache with,
                 simulated on the same routing (miss rates only).

Sources (the pages' titles):
* "FreeToken: Efficient Edge-Native MoE Serving with Bandwidth-Adaptive
  Execution" (paper summary) - design paragraph: full expert pool in host
  memory, a GPU expert cache shared by all MoE layers with slots keyed by
  (layer, expert); routing dedup, hit classification and LRU victim selection
  in one GPU kernel; the cache rebuilt at scheduler safe points when the VRAM
  budget changes; ablation paragraph: global LRU, double buffering.
* "FreeToken vs vLLM on one RTX 3090: BF16 MoE RAM offload compared" - Runtime
  configurations (slot cache with LRU replacement) and "Why the performance
  differs" (256 routed experts, eight selected per token, the bank kept in
  host memory, selected experts fetched on demand).
* "FreeToken: az VRAM ile büyük MoE modelleri" - intro (experts in host RAM,
  LRU expert cache on the GPU, misses streamed over PCIe) and the "Tuzaklar"
  printout naming the fp8_block weight format.

Parity status: every function here is pinned by the CPU tests in
``tests/test_oracle_*.py`` (brute-force replays, closed forms, invariants,
library cross-checks).  The pages print no worked example of routing, cache
or FFN values, so no pin compares against a printed value except the
expert-size arithmetic in ``tests/golden/page_sizes.txt``.
"""

from . import cache, ffn, fp8, routing, stream  # noqa: F401
