"""Host-side parts of bench.py that need no GPU: the oracle's CPU baseline
(all host cores, then one thread) on a tiny workload."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402


def test_cpu_baseline_times_all_cores_and_one_thread():
    w = bench.workload_by_name("er5k-tiny")
    part = w.make(bench.SEED)
    n_before = oracle.num_threads()
    cpu = bench.cpu_baseline_entry(part, w, 0.2)
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] == n_before
    one = cpu["single_thread"]
    assert one["value"] > 0 and one["unit"] == cpu["unit"]
    assert "1 OpenMP threads" in one["sample"]
    assert oracle.num_threads() == n_before  # restored


def test_oracle_thread_count_can_be_set_and_restored():
    n = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        assert oracle.num_threads() == 1
    finally:
        oracle.set_num_threads(n)
    assert oracle.num_threads() == n
