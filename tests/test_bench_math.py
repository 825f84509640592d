"""CPU checks of the bench's derived measurements: the marginal host-link fit
and the per-launch HBM-or-link bound (bench.py), on synthetic launch data
whose answer is known, and the in-pipeline DRAM traffic scaled from a small
capture."""
import sys

import numpy as np
import pytest


@pytest.fixture(scope="module")
def bench():
    saved = sys.argv
    sys.argv = ["bench.py"]
    try:
        import bench as b
    finally:
        sys.argv = saved
    return b


def test_marginal_link_recovers_slope_and_intercept(bench):
    eb = 6_291_456
    rng = np.random.default_rng(3)
    carried = rng.integers(0, 5, size=400)
    per_blob_ms, alone_ms = eb / 240e9 * 1e3, 0.0225        # 240 GB/s, 22.5 us
    window = alone_ms + per_blob_ms * carried + rng.normal(0, 1e-4, size=carried.size)
    m = bench.marginal_link(carried, window, eb)
    assert m["gbs"] == pytest.approx(240.0, rel=0.02)
    assert m["intercept_us"] == pytest.approx(22.5, abs=0.2)
    assert sum(m["launches_by_blobs_copied"].values()) == carried.size


def test_marginal_link_needs_two_copy_counts(bench):
    assert bench.marginal_link(np.zeros(10), np.ones(10), 1) is None


def test_bound_takes_the_slower_resource_per_launch(bench):
    eb = 1e9                                                  # 1 GB blobs: easy arithmetic
    nuniq = np.array([8.0, 8.0, 1.0])
    carried = np.array([0.0, 1.0, 4.0])
    window_ms = np.array([2.0, 10.0, 40.0])
    b = bench.bound_of_launches((nuniq, carried, window_ms), eb, hbm_gbs=8000.0, link_gbs=200.0)
    # launch bounds: 8 GB / 8000 GB/s = 1 ms; max(1 ms, 1 GB / 200 GB/s = 5 ms); max(0.125, 20) ms
    assert b["bound_us_per_launch"] == pytest.approx((1000 + 5000 + 20000) / 3)
    assert b["measured_us_per_launch"] == pytest.approx((2 + 10 + 40) / 3 * 1000)
    assert b["link_bound_launches"] == pytest.approx(2 / 3)
    assert bench.bound_of_launches(None, eb, 8000.0, 200.0) is None
    assert bench.bound_of_launches((nuniq, carried, window_ms), eb, 8000.0, None) is None


def test_pipeline_traffic_scales_the_small_capture_by_unique_experts(bench):
    per_unique, writes = bench.FFN_PIPELINE_TRAFFIC["qwen35b-a3b-shape-decode-b1"]
    # the capture read each launch's 8 experts once: about 6.3 MB per unique expert
    assert per_unique == pytest.approx(6291456 * 1.0017, rel=1e-3)
    assert bench.pipeline_traffic("qwen35b-a3b-shape-decode-b1", 8.0) == pytest.approx(8 * per_unique + writes)
    assert bench.pipeline_traffic("qwen35b-a3b-shape-decode-b1", 4.0) < bench.pipeline_traffic(
        "qwen35b-a3b-shape-decode-b1", 8.0)
    assert bench.pipeline_traffic("no-such-workload", 8.0) is None
