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


def _simulated_floor(part, counts_source, rb, streamed, n_rows, k_rows):
    """DRAM bytes of one launch under a static cache of the k_rows most gathered
    rows, by walking the gathers in order: a cached row is read at its first
    gather, any other row at every gather; a row never gathered is read once
    (the compulsory bytes read every input row)."""
    import numpy as np

    counts = np.bincount(counts_source, minlength=n_rows)
    cached = set(np.argsort(-counts, kind="stable")[:k_rows].tolist())
    seen, reads = set(), 0
    for c in counts_source.tolist():
        if c not in seen or c not in cached:
            reads += rb
        seen.add(c)
    return streamed + reads + (n_rows - len(seen)) * rb


def test_cache_floor_matches_a_simulated_static_cache():
    # the roofline's cache-aware bytes against a gather-by-gather walk of the same partition
    import numpy as np

    w = bench.workload_by_name("rmat16m-tiny")
    part = w.make(bench.SEED)
    elem, gel = 2, 4
    fwd_b, bwd_b = bench.aggregation_bytes(part, w, elem, grad_elem=gel)
    nT, nL = part.n_total, part.n_local
    row_of = np.repeat(np.arange(nL), np.diff(part.rowptr))  # the backward gathers row v once per entry of row v
    for k_rows in (0, 37, 500, 10 ** 9):
        l2 = [k_rows * w.widths[l] * elem for l in range(w.layers)]
        for l in range(w.layers):
            rb = w.widths[l] * elem
            got = bench.cache_floor_bytes(part, w, elem, gel, l2[l])[l]
            streamed = fwd_b[l] - nT * rb
            assert got == _simulated_floor(part, part.colidx, rb, streamed, nT, min(k_rows, nT)), (k_rows, l)
        for i, l in enumerate(range(w.layers - 1, 0, -1)):
            rb = w.widths[l] * gel
            got = bench.cache_floor_bytes(part, w, elem, gel, k_rows * rb)[w.layers + i]
            streamed = bwd_b[i] - nL * rb
            assert got == _simulated_floor(part, row_of, rb, streamed, nL, min(k_rows, nL)), (k_rows, l)
    # no cache: every gather from DRAM; an unbounded cache: the compulsory bytes
    none = bench.cache_floor_bytes(part, w, elem, gel, 0)
    full = bench.cache_floor_bytes(part, w, elem, gel, 1 << 62)
    assert full == fwd_b + bwd_b
    gathered = np.unique(part.colidx).shape[0]
    assert none[0] == fwd_b[0] - nT * w.widths[0] * elem + (part.nnz + nT - gathered) * w.widths[0] * elem


def test_reference_arm_prints_the_contract_line(capsys):
    # the oracle arm on a tiny workload: one JSON line with the contract's keys and the oracle as its baseline
    import json

    bench.main(["--impl", "reference", "--workload", "er5k-tiny", "--steps", "2", "--warmup", "1",
                "--ref-seconds", "0.05"])
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "er5k-tiny"
