"""Host logic of bench.py on CPU: the algorithmic byte counts behind the
roofline figure, and the lookup of the captured DRAM traffic."""
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import synthetic  # noqa: E402


def _batch(temperatures, gamma=5, V=64):
    w = synthetic.WORKLOADS[4].variant(B=len(temperatures), gamma=gamma, V=V)
    batch = synthetic.generate(w, seed=3)
    batch.temperature[:] = np.asarray(temperatures, np.float32)
    return batch


def _rows_read(batch, n):
    """Rows of logits the full read touches, counted request by request."""
    G = batch.workload.gamma
    rows = 0
    for b in range(batch.B):
        T = float(batch.temperature[b])
        sampled = 0.0 < T < float("inf")
        rows += G + 1                      # every target row is streamed
        if sampled:
            rows += G                      # and every draft row of a sampled request
            if n[b] >= 0:
                rows += 2 if n[b] < G else 1  # the draw re-reads its row(s)
    return rows


def test_full_read_counts_every_streamed_row():
    G = 5
    T = [0.0, 0.7, 1.0, float("inf"), float("nan"), 0.3, 0.0, 2.0]
    batch = _batch(T, gamma=G)
    n = np.array([G, 0, G, 2, -1, -1, 3, 4], np.int32)
    w = batch.workload
    small = batch.B * G * 8 + batch.B * 12 + batch.B * (G + 1) * 4
    assert bench.algorithmic_bytes(batch, n) == w.elem_bytes * w.V * _rows_read(batch, n) + small


def test_early_exit_never_reads_more_than_the_full_read():
    G = 6
    rng = np.random.default_rng(11)
    for _ in range(20):
        T = rng.choice([0.0, 0.3, 1.0], size=10)
        batch = _batch(T, gamma=G)
        n = rng.integers(0, G + 1, size=10).astype(np.int32)
        assert bench.algorithmic_bytes_early(batch, n) <= bench.algorithmic_bytes(batch, n)


@pytest.mark.parametrize("T", [0.0, 0.8])
def test_early_exit_equals_the_full_read_when_every_proposal_is_accepted(T):
    G = 4
    batch = _batch([T] * 6, gamma=G)
    n = np.full(6, G, np.int32)
    assert bench.algorithmic_bytes_early(batch, n) == bench.algorithmic_bytes(batch, n)


def test_captured_traffic_is_keyed_by_workload_and_early_exit(tmp_path):
    h = bench.kernel_hash()
    prof = {"mixed": {"kernel_hash": h, "dram_bytes_per_launch": 11.0},
            "large-early": {"kernel_hash": h, "dram_bytes_per_launch": 22.0},
            "sampling": {"kernel_hash": "0" * 16, "dram_bytes_per_launch": 33.0}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(prof))
    assert bench.captured_traffic("mixed", False, str(path)) == 11.0
    assert bench.captured_traffic("large", True, str(path)) == 22.0
    assert bench.captured_traffic("large", False, str(path)) is None   # the full read was not captured
    assert bench.captured_traffic("mixed", True, str(path)) is None    # nor early exit on this workload
    assert bench.captured_traffic("sampling", False, str(path)) is None  # captured from other sources
    assert bench.captured_traffic("mixed", False, str(tmp_path / "missing.json")) is None


def test_kernel_hash_covers_existing_sources():
    for rel in bench.KERNEL_SOURCES:
        assert os.path.isfile(os.path.join(ROOT, rel)), rel
    assert len(bench.kernel_hash()) == 16
    # each kernel is keyed on its own source: the streaming and early-exit
    # kernels share one, the one-block and cluster kernels have their own
    assert bench.kernel_hash("early_kernel<bf16>") == bench.kernel_hash("stream_kernel<f32>")
    assert len({bench.kernel_hash(k) for k in ("stream_kernel", "rowwise_kernel", "cluster_kernel")}) == 3


def test_captured_traffic_uses_the_entry_kernels_sources(tmp_path):
    prof = {"greedy": {"kernel": "cluster_kernel<bf16, 16>", "kernel_hash": bench.kernel_hash("cluster_kernel"),
                       "dram_bytes_per_launch": 44.0},
            "tiny": {"kernel": "rowwise_kernel<f32>", "kernel_hash": bench.kernel_hash("stream_kernel"),
                     "dram_bytes_per_launch": 55.0}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(prof))
    assert bench.captured_traffic("greedy", False, str(path)) == 44.0
    assert bench.captured_traffic("tiny", False, str(path)) is None  # keyed on another kernel's sources
