"""Pins of the oracle's top-k selection and gate weights.

Each check ties the oracle to something other than its own code: a brute
force scan written here, numpy's stable argsort, scipy's softmax, closed forms.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

import synth
from oracle import routing


def brute_topk(row, k):
    """Repeatedly scan for the largest remaining logit; the first (lowest index) wins ties."""
    vals = [(-math.inf if math.isnan(v) else float(v)) for v in row]
    taken, out = set(), []
    for _ in range(k):
        best = None
        for e, v in enumerate(vals):
            if e in taken:
                continue
            if best is None or v > vals[best]:
                best = e
        taken.add(best)
        out.append(best)
    return out


@pytest.mark.parametrize("E,k", [(16, 2), (256, 8), (64, 6), (8, 8)])
def test_topk_matches_brute_force_random(E, k):
    lg = synth.normal(synth.key(5, E, k), 40 * E).reshape(40, E)
    got = routing.topk(lg, k)
    for t in range(lg.shape[0]):
        assert got[t].tolist() == brute_topk(lg[t], k)


@pytest.mark.parametrize("E,k", [(16, 2), (256, 8), (32, 5)])
def test_topk_tie_heavy_matches_stable_argsort(E, k):
    lg = synth.router_ties(11, E * k, (200, E))
    assert len(np.unique(lg)) < 40               # many ties by construction
    got = routing.topk(lg, k)
    ref = np.argsort(-lg.astype(np.float64), axis=-1, kind="stable")[:, :k]
    np.testing.assert_array_equal(got, ref)
    for t in range(0, 200, 17):
        assert got[t].tolist() == brute_topk(lg[t], k)


def test_signed_zero_and_nan_ordering():
    row = np.array([-0.0, 0.0, np.nan, -1.0, 0.0, np.nan], dtype=np.float32)
    # +-0 tie -> index order 0,1,4; then -1 (index 3); then NaN as -inf by index 2, 5
    assert routing.topk(row[None], 6)[0].tolist() == [0, 1, 4, 3, 2, 5]
    assert routing.topk(row[None], 6)[0].tolist() == brute_topk(row, 6)


def test_gates_closed_forms():
    # equal selected logits -> uniform gates
    lg = np.array([[1.0, 1.0, 1.0, 1.0, -3.0]], dtype=np.float32)
    idx, w = routing.route(lg, 4)
    assert idx[0].tolist() == [0, 1, 2, 3]
    np.testing.assert_allclose(w, 0.25, rtol=0, atol=1e-15)
    # two picks with logit gap d -> logistic(d)
    d = 1.25
    idx, w = routing.route(np.array([[0.0, d, -5.0]], dtype=np.float32), 2)
    assert idx[0].tolist() == [1, 0]
    assert abs(w[0, 0] - 1.0 / (1.0 + math.exp(-d))) < 1e-15
    # k = 1 -> gate exactly 1
    idx, w = routing.route(np.array([[0.3, 2.0, -1.0]], dtype=np.float32), 1)
    assert w[0, 0] == 1.0


@pytest.mark.parametrize("E,k", [(16, 2), (256, 8)])
def test_gates_equal_full_softmax_renormalised(E, k):
    lg = synth.normal(synth.key(9, E), 64 * E).reshape(64, E)
    idx, w = routing.route(lg, k)
    full = softmax(lg.astype(np.float64), axis=-1)
    sel = np.take_along_axis(full, idx.astype(np.int64), axis=-1)
    np.testing.assert_allclose(w, sel / sel.sum(-1, keepdims=True), rtol=1e-13, atol=0)
    np.testing.assert_allclose(w.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(w, axis=-1) <= 0)         # selection order = descending gate
