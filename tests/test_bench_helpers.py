"""Host-side helpers of bench.py (no GPU): sample indices, the clock-sample
time stamps, the scaled DRAM traffic, the host core description."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_sample_indices_cover_every_chunk_edge_of_the_torus():
    w = synth.WORKLOADS["torus4x4_lm300m"]
    idx = bench.sample_indices(w, [(0, w.N)], n_rand=100)
    assert idx.min() >= 0 and idx.max() < w.N and np.all(np.diff(idx) > 0)
    # row chunk c starts at c*N/4; its sub-chunk d at c*N/4 + d*N/16 (N divisible by 16)
    for c in range(4):
        for d in range(4):
            e = c * (w.N // 4) + d * (w.N // 16)
            for q in (e - 1, e):
                if 0 <= q < w.N:
                    assert q in set(idx.tolist()), q


def test_sample_indices_multiring_buckets_and_small_buffers():
    w = synth.WORKLOADS["multiring64_resnet101"]
    buckets = [(w.N - 1000, w.N), (0, w.N - 1000)]
    idx = set(bench.sample_indices(w, buckets, n_rand=10).tolist())
    # slice edges of the top bucket (k = 4 slices of 250) and its first chunk edges
    for e in (w.N - 1000, w.N - 750, w.N - 500, w.N - 250, w.N - 1000 + 4):
        assert e in idx, e
    small = synth.WORKLOADS["ring4_int"]
    assert np.array_equal(bench.sample_indices(small, [(0, small.N)]), np.arange(small.N))


def test_clock_stamp_keeps_milliseconds():
    a = bench.ClockSampler._stamp("2026/12/03 05:29:46.125")
    b = bench.ClockSampler._stamp("2026/12/03 05:29:46")
    assert abs((a - b) - 0.125) < 1e-9


def test_traffic_scales_with_the_launch_bytes(monkeypatch):
    w = synth.WORKLOADS["torus4x4_resnet50"]
    monkeypatch.setattr(bench, "kernel_hash", lambda: "feedfacefeedface")
    monkeypatch.setitem(bench.NCU_TRAFFIC, ("torus", "f32", "ldg", "feedfacefeedface"), (900, 1000))
    assert bench.ncu_traffic(w, "auto", 2000) == 1800
    assert bench.ncu_traffic(w, "chunked", 2000) is None
    assert bench.ncu_traffic(w.with_(dtype="f16"), "auto", 2000) is None


def test_host_cpu_reports_cores_and_model():
    h = bench.host_cpu()
    assert h["nproc"] >= 1 and isinstance(h["cpu_model"], str) and h["cpu_model"]
