"""Pin the oracle's expert-blob size arithmetic to the sizes the pages print.

The pages print no worked routing / cache / FFN values; what they do print
(host bank size, fp8 bank size, slot count in a VRAM budget) fixes how many
bytes one (layer, expert) blob holds.  Fixture: tests/golden/page_sizes.txt.
"""
import os

from oracle import ffn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_sizes.txt")
GIB = 1024 ** 3
L, E, H, I = 40, 256, 2048, 512


def load():
    out = {}
    for line in open(GOLDEN, encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        name, value, unit, tol, _src = [p.strip() for p in line.split("|", 4)]
        out[name] = (float(value), unit, float(tol))
    return out


def test_bf16_bank_matches_host_memory_growth():
    g = load()
    bank = L * E * ffn.expert_bytes(H, I, ffn.W_BF16)
    v, unit, tol = g["bf16_bank_host_increase"]
    assert unit == "GiB" and abs(bank / GIB - v) <= tol * v
    v, _, _ = g["bf16_checkpoint_upper_bound"]
    assert bank / GIB < v                      # experts are part of the checkpoint
    assert v - bank / GIB < 10                 # and most of it


def test_fp8_bank_matches_printed_size():
    v, unit, tol = load()["fp8_bank"]
    bank = L * E * ffn.expert_bytes(H, I, ffn.W_FP8)
    assert unit == "GB" and abs(bank / 1e9 - v) <= tol * v


def test_auto_cache_fits_the_vram_budget():
    g = load()
    slots, _, _ = g["bf16_auto_cache_slots"]
    vram, _, _ = g["bf16_vram_used"]
    cache = slots * ffn.expert_bytes(H, I, ffn.W_BF16) / GIB
    assert cache < vram and vram - cache < 10  # the rest: ~3 GiB non-expert weights + KV + workspace
