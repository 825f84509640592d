"""The bounds-checked build of libft (-DFT_CHECKED) on the GPU.

In that build every kernel checks the table and plan indices it dereferences
(slot, key, expert, row and offset indices); an index out of range raises
FT_ERR_CHECKED in the cache's sticky status and the access is skipped, so a
corrupted table is reported instead of read or written out of range.  The
checks stand in for a memory checker, which this GPU pool does not offer.

1. On valid tables the checks raise nothing: decode (fused and two-kernel
   FFN, SM pull and copy engine, step-graph replay), a resize, and prefill
   (bf16 and fp8) through the checked library match the oracle as the normal
   build does.
2. A slot-table entry overwritten with a slot outside [0, C) (or below -1) is
   reported as FT_ERR_CHECKED by the next synchronous call.  Only the routing
   kernel reads the slot table as an index, and in this build it reads such an
   entry as "absent" after reporting it, so no kernel touches memory out of
   range.  A new cache afterwards works.

Each case runs in a child process, because a process loads one build of the
library (FT_CHECKED=1 selects the checked one).
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_checked(code: str, timeout: int = 900) -> str:
    env = dict(os.environ, FT_CHECKED="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=timeout)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return r.stdout


PARITY = r"""
import expert_cache_host_layer_gb300 as ft
assert ft.ft_checked_build() and "_build_checked" in ft.LIB_PATH
from synth import workloads as W
from tests.harness import run_parity, run_parity_graph
from tests.test_gpu_prefill import FP8_SMALL_PREFILL
q = W.QWEN35B_DECODE.replace(num_layers=4, num_slots=96)
for name, rep in [
    ("tiny sm-pull", run_parity(W.TINY, steps=16)),
    ("tiny copy-engine", run_parity(W.TINY, steps=16, fetch_mode=0)),
    ("tiny resize", run_parity(W.TINY.replace(resize_step=8, resize_slots=8), steps=16)),
    ("35b b1", run_parity(q, steps=12, bank_blobs=256)),
    ("35b b4", run_parity(q.replace(tokens=4), steps=6, bank_blobs=256)),
    ("35b b1 graph", run_parity_graph(q, steps=6, bank_blobs=256)),
    ("prefill 200", run_parity(W.QWEN35B_PREFILL.replace(num_layers=2, tokens=200), steps=1, bank_blobs=512)),
    ("fp8 prefill", run_parity(FP8_SMALL_PREFILL, steps=1)),
]:
    assert rep["events"] > 0 and rep["ffn_checked"] > 0, (name, rep)
    print(name, rep["events"], rep["ffn_checked"], rep["max_err"])
print("checked parity ok")
"""


def test_checked_build_matches_the_oracle():
    out = run_checked(PARITY)
    assert "checked parity ok" in out
    print(out)


CORRUPT = r"""
import torch
import expert_cache_host_layer_gb300 as ft
from expert_cache_host_layer_gb300.pipeline import ExpertCache
from synth import workloads as W
from tests.harness import make_bank, run_parity
assert ft.ft_checked_build()
w = W.TINY
bank, n_blobs = make_bank(w)
dev = torch.device("cuda:0")
E = w.num_experts
for bad in (w.num_slots, w.num_slots + 7, -5, 2 ** 30):
    c = ExpertCache(w.num_layers, E, w.top_k, w.hidden, w.inter, w.wdtype, w.num_slots, 1, bank, n_blobs,
                    fetch_mode=1, device=dev)
    x = torch.zeros((1, w.hidden), dtype=c.act_dtype, device=dev)
    y = torch.empty((1, w.hidden), dtype=c.out_dtype, device=dev)
    lg = torch.full((1, E), -1.0, dtype=torch.float32, device=dev)
    lg[0, 3], lg[0, 9] = 5.0, 4.0   # experts 3 and 9 at every layer
    for layer in range(w.num_layers):
        c.route_classify(layer, lg); c.fetch_misses(layer); c.moe_forward(layer, x, y)
    c.synchronize()
    assert c.tables()[0][3] >= 0   # (layer 0, expert 3) is cached
    ft.ft_debug_set_key_slot(c.handle, 3, bad)
    c.route_classify(0, lg)
    try:
        c.synchronize()
        raise AssertionError("no FT_ERR_CHECKED for slot %d" % bad)
    except ft.FtError as ex:
        assert ex.status == ft.FT_ERR_CHECKED, ex
    c.close()
    print("slot", bad, "reported")
rep = run_parity(w, steps=8)   # a new cache afterwards works
assert rep["events"] == 8 * w.num_layers
print("corrupt slot ok")
"""


def test_out_of_range_slot_is_reported_not_dereferenced():
    out = run_checked(CORRUPT)
    assert "corrupt slot ok" in out
    print(out)


def test_normal_build_refuses_the_corrupting_knob():
    import torch

    import expert_cache_host_layer_gb300 as ft
    from expert_cache_host_layer_gb300.pipeline import ExpertCache
    from synth import workloads as W
    from tests.harness import make_bank
    if ft.ft_checked_build():
        pytest.skip("this process loaded the checked build")
    w = W.TINY
    bank, n_blobs = make_bank(w)
    c = ExpertCache(w.num_layers, w.num_experts, w.top_k, w.hidden, w.inter, w.wdtype, w.num_slots, 1, bank,
                    n_blobs, fetch_mode=1, device=torch.device("cuda:0"))
    try:
        with pytest.raises(ft.FtError) as ei:
            ft.ft_debug_set_key_slot(c.handle, 3, w.num_slots + 7)
        assert ei.value.status == ft.FT_ERR_STATE
    finally:
        c.close()
