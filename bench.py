#!/usr/bin/env python
"""Benchmark of the hot path: one full-graph training epoch of one graph partition.

A step is one epoch on one partition through the C ABI: for every layer a halo
pull from the stale-representation table, the forward aggregation and update,
the push of the new local rows; the softmax-CE gradient; for every layer the
backward update and (past the first layer) the backward aggregation with the
halo-row gradients.  The metric is aggregated edge x feature per second: the
sum over the step's aggregations of (entries x feature width), divided by the
step time.

Default workload: one partition of an R-MAT scale-24 graph (8,388,608 local +
4,194,304 halo vertices, ~408M local entries with self loops), 3-layer GCN
128 -> 256 -> 256 -> 172, bf16 storage with fp32 accumulation, stale tables of
2^24 rows.  All inputs are synthetic and seeded (synth/).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

With N > 1 the script runs under torchrun, one partition per rank (weak
scaling, no data-path collective); timing is the max over ranks.
``--impl reference`` times the CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth.configs import PROFILE, TINY, WORKLOADS  # noqa: E402

METRIC = "GCN layer fwd+bwd: edge·feat/s, epoch ms, % HBM roofline (SpMM) / % TC peak"
UNIT = "edge*feat/s"
SEED = 0


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------

def rank_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def init_dist(world: int, use_cuda: bool):
    if world <= 1:
        return None
    import torch.distributed as dist

    dist.init_process_group(backend="nccl" if use_cuda else "gloo")
    return dist


def barrier(dist, use_cuda: bool):
    if dist is None:
        return
    if use_cuda:
        import torch

        dist.barrier(device_ids=[torch.cuda.current_device()])
    else:
        dist.barrier()


def max_over_ranks(dist, x: float, use_cuda: bool) -> float:
    """Max of a host scalar over all ranks (identity for a single process)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if use_cuda else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, x: float, use_cuda: bool) -> float:
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if use_cuda else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def workload_by_name(name: str):
    if name.endswith("-tiny"):
        return TINY[name[:-5]]
    if name in PROFILE:
        return PROFILE[name]
    return WORKLOADS[name]


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def edge_feat_per_step(part, w) -> int:
    """Entries x feature width summed over the step's aggregations of the layer in
    its textbook order (forward on every layer at its input width; backward, over
    the transpose, on every layer but the first): a fixed property of the workload,
    whatever order the library multiplies in."""
    fwd = sum(part.nnz * f for f in w.widths[:-1])
    bwd = sum(part.nnz * f for f in w.widths[1:-1])
    return int(fwd + bwd)


def narrow_layers(w, enabled: bool = False):
    """Layers the partition model runs with the multiplication first (--narrow: GCN, output narrower than input)."""
    return [enabled and w.agg != "sage" and w.widths[l + 1] < w.widths[l] for l in range(w.layers)]


def aggregation_bytes(part, w, elem: int, narrow: bool = False, grad_elem: int = None):
    """Compulsory bytes of each aggregation launch of one step, in launch order
    (forward layers 0..L-1, then backward layers L-1..1): row pointers, column
    ids, the normalisation vector, every input row once and every output row once.
    The backward launches move gradient rows (grad_elem bytes per value, default
    elem).  A narrow layer aggregates at its output width (T = H W forward, dY
    backward), and its backward aggregation also runs on the first layer."""
    gel = elem if grad_elem is None else grad_elem
    nL, nT, nnz = part.n_local, part.n_total, part.nnz
    sage = w.agg == "sage"
    nar = narrow_layers(w, narrow)
    fwd, bwd = [], []
    for l in range(w.layers):
        f = w.widths[l + 1] if nar[l] else w.widths[l]
        out_cols = 2 * f if sage else f
        fwd.append(4 * (nL + 1) + 4 * nnz + 4 * (nL if sage else nT) + nT * f * elem + nL * out_cols * elem)
    for l in range(w.layers - 1, -1, -1):
        if l == 0 and not nar[l]:
            continue
        f = w.widths[l + 1] if nar[l] else w.widths[l]
        in_cols = 2 * f if sage else f
        bwd.append(4 * (nT + 1) + 4 * nnz + 4 * (nL if sage else nT) + nL * in_cols * gel + nT * f * gel)
    return fwd, bwd


def cache_floor_bytes(part, w, elem: int, grad_elem: int, l2_bytes: int, narrow: bool = False):
    """DRAM bytes of one step's aggregation launches under an ideal static cache
    of l2_bytes: the most-gathered rows that fit stay resident (each read once),
    every other gather goes to DRAM, and the streamed terms of the compulsory
    bytes (row pointers, column ids, normalisation, outputs) are read or written
    once.  For the power-law gathers here this is the reachable floor of a
    kernel that cannot reorder its gathers; the compulsory bytes assume an
    infinite cache."""
    import numpy as np

    fwd_b, bwd_b = aggregation_bytes(part, w, elem, narrow, grad_elem)
    nT = part.n_total
    col_counts = np.sort(np.bincount(part.colidx, minlength=nT))[::-1]  # forward: gathers of each input row
    row_counts = np.sort(np.diff(part.rowptr).astype(np.int64))[::-1]   # backward: gathers of each dZ row
    nar = narrow_layers(w, narrow)
    sage = w.agg == "sage"

    def floor(counts, rb, compulsory):
        # the compulsory bytes read every input row once; a row outside the
        # cache is read again for each of its gathers after the first
        k = max(0, min(len(counts), int(l2_bytes // rb)))
        rest = counts[k:]
        return compulsory + int(np.maximum(rest - 1, 0).sum()) * rb

    out = []
    for l, b in zip(range(w.layers), fwd_b):
        f = w.widths[l + 1] if nar[l] else w.widths[l]
        out.append(floor(col_counts, f * elem, b))
    bl = [l for l in range(w.layers - 1, -1, -1) if not (l == 0 and not nar[l])]
    for l, b in zip(bl, bwd_b):
        f = w.widths[l + 1] if nar[l] else w.widths[l]
        rb = (2 * f if sage else f) * grad_elem
        out.append(floor(row_counts, rb, b))
    return out


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1939.4)), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha1()
    for name in ("aggregate.cu", "setup.cu"):  # the kernel, and the entry order and tiers it streams
        h.update(open(os.path.join(ROOT, "sparse_aggregation_dense_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:12]


def small_case_traffic():
    """Per-launch DRAM bytes of the aggregation on the quarter-size R-MAT case
    (rmat4m) from the committed ncu summary, if it was taken on the current
    kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "aggregate_rmat4m.md")
    if not os.path.exists(p):
        return None
    src, rows = None, []
    for line in open(p):
        if line.startswith("kernel_source_sha1:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("launch:"):
            name, gb, ms = [x.strip() for x in line.split(":", 1)[1].split(",")]
            rows.append({"launch": name, "dram_gb": float(gb), "ncu_ms": float(ms),
                         "dram_gbs": round(float(gb) / float(ms) * 1e3, 1)})
    if src != kernel_source_hash() or not rows:
        return None
    return {"workload": "rmat4m", "launches": rows, "note": "one step's five aggregation launches under ncu "
            "(serialised; DRAM bytes per launch); the full-size step is not captured with counters"}


def ncu_traffic(workload: str, grad: str):
    """DRAM bytes of one step's aggregation launches from the committed ncu
    summary, if it was taken on the current kernel source with the same gradient
    storage; else None."""
    p = os.path.join(ROOT, "profiles", f"aggregate_{workload}.txt")
    if not os.path.exists(p):
        return None
    src, traffic, gd = None, None, None
    for line in open(p):
        if line.startswith("kernel_source_sha1:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_step_aggregations:"):
            traffic = float(line.split(":", 1)[1].strip())
        if line.startswith("grad_dtype:"):
            gd = line.split(":", 1)[1].strip()
    if src != kernel_source_hash() or traffic is None or gd != grad:
        return None
    return traffic


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.remove(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def oracle_sample(part, w, target_s: float, seed: int, batch_rows: int = 4096, max_batches: int = 64):
    """Time the oracle on row samples of one epoch until about target_s seconds of
    oracle work; returns (edge_feat, seconds, description).

    A batch holds, for every layer, the forward aggregation + update + update
    backward of `batch_rows` random local rows and, past the first layer, the
    backward aggregation of a proportional number of random transpose rows.
    Input preparation (generator calls, widening, the sampled sub-transpose) is
    not timed."""
    import oracle

    bf = w.dtype == "bf16"
    nL, nT = part.n_local, part.n_total
    sage = w.agg == "sage"
    wts = oracle.sage_invcnt(part) if sage else oracle.gcn_dinv(part)
    rows_t = min(nT, max(1, batch_rows * nT // max(nL, 1)))
    deg = np.diff(part.rowptr)
    # sampled transpose rows for every batch, and the block entries they hold
    U_all = synth.sample_rows(nT, rows_t * max_batches, seed + 77)
    rng = np.random.default_rng(seed)
    U_all = U_all[rng.permutation(U_all.shape[0])]
    sel = np.zeros(nT, bool)
    sel[U_all] = True
    keep = sel[part.colidx]
    row_of = np.repeat(np.arange(nL), deg)
    cnt = np.bincount(row_of[keep], minlength=nL)
    sub = synth.Partition(np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32), part.colidx[keep], nL,
                          part.n_halo, part.deg, part.local_ids, part.halo_ids, part.n_table)
    T = oracle.transpose(sub)
    del keep, row_of
    ef, secs, batches = 0, 0.0, 0
    while batches < max_batches and secs < target_s:
        b = batches
        for l in range(w.layers):
            f_in, f_out = w.widths[l], w.widths[l + 1]
            K = 2 * f_in if sage else f_in
            rows = synth.sample_rows(nL, batch_rows, seed + 1000 * b + l)
            parts = [part.colidx[part.rowptr[r]:part.rowptr[r + 1]] for r in rows]
            cols = np.unique(np.concatenate(parts + [rows.astype(np.int32)]).astype(np.int64))
            hmap = -np.ones(nT, np.int64)
            hmap[cols] = np.arange(cols.shape[0])
            Hs = oracle.widen(synth.features(0, f_in, f_in, SEED, 900 + l, bf16=bf, ids=cols), bf)
            W = synth.glorot(K, f_out, SEED, synth.STREAM_WEIGHT + l).astype(np.float64)
            G = oracle.widen(synth.features(rows.shape[0], f_out, f_out, SEED, 950 + l, bf16=bf), bf)
            relu = l < w.layers - 1
            t0 = time.perf_counter()
            Z = oracle.aggregate(part, Hs, f_in, w.agg, rows=rows, hmap=hmap, weights=wts)
            Ho = oracle.update(Z, W, relu)
            oracle.update_backward(G, Ho, Z, W, relu, want_dz=l > 0)
            secs += time.perf_counter() - t0
            ef += int(deg[rows].sum()) * f_in
            del Hs, hmap, Z, Ho, G
            if l == 0:
                continue
            U = U_all[b * rows_t:(b + 1) * rows_t]
            V = np.unique(np.concatenate([T[1][T[0][u]:T[0][u + 1]] for u in U] + [np.zeros(0, np.int32)]))
            V = V.astype(np.int64)
            vmap = -np.ones(nL, np.int64)
            vmap[V] = np.arange(V.shape[0])
            width = 2 * f_in if sage else f_in
            dZ = oracle.widen(synth.features(0, width, width, SEED, 980 + l, bf16=bf, ids=V), bf)
            t0 = time.perf_counter()
            oracle.aggregate_backward(part, T, dZ, f_in, w.agg, rows=U, dmap=vmap, weights=wts)
            secs += time.perf_counter() - t0
            ef += int(np.diff(T[0])[U].sum()) * f_in
            del dZ, vmap
        batches += 1
    desc = (f"{batches} batches; each: {batch_rows} random local rows per layer (forward aggregation + update + "
            f"update backward) and {rows_t} random transpose rows per layer past the first (backward aggregation); "
            f"double precision, {oracle.num_threads()} OpenMP threads; input preparation not timed")
    return ef, secs, desc


def cpu_baseline_entry(part, w, seconds: float):
    """The oracle on all host cores (about `seconds` of work) and, on a quarter of
    that, on one thread."""
    import oracle

    cef, csec, desc = oracle_sample(part, w, seconds, SEED)
    cpu = {"value": cef / csec, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle", "sample": desc,
           "seconds": round(csec, 2)}
    n_all = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        sef, ssec, sdesc = oracle_sample(part, w, seconds / 4, SEED + 5, max_batches=16)
    finally:
        oracle.set_num_threads(n_all)
    cpu["single_thread"] = {"value": sef / ssec, "unit": UNIT, "seconds": round(ssec, 2), "sample": sdesc}
    return cpu


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

def fill_table(tab, n_rows, f, bf, seed, stream, dist, chunk=1 << 20):
    """Generate a table on the host in chunks and copy it to the device view."""
    import torch

    ld = tab.stride(0)
    buf = tab.as_strided((n_rows, ld), (ld, 1))
    for r0 in range(0, n_rows, chunk):
        n = min(chunk, n_rows - r0)
        ids = np.arange(r0, r0 + n, dtype=np.int64)
        h = synth.features(0, f, ld, seed, stream, dist, bf16=bf, ids=ids)
        t = torch.from_numpy(h.view(np.int16) if bf else h)
        if bf:
            t = t.view(torch.bfloat16)
        buf[r0:r0 + n].copy_(t, non_blocking=False)



def measure_codec(m, part, w, tdt, stream, reps: int = 5):
    """Low-bit halo codec (Sylvie Quantizer / Dequantizer) on the layer-1 rows of the partition: the quantising
    push of all local rows and the dequantising pull of all halo rows, per bit width, against the plain
    push / pull of the same rows.  Bytes are the compulsory ones (row data, ids, scale / zero point)."""
    import torch

    from sparse_aggregation_dense_gb300 import gnn

    f, es = w.widths[1], (2 if tdt == torch.bfloat16 else 4)
    nL, nH, nT = part.n_local, part.n_halo, part.n_table
    H = m.H[1]
    lid = torch.from_numpy(part.local_ids).cuda()
    hid = torch.from_numpy(part.halo_ids).cuda()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        ev[0].record(stream)
        for _ in range(reps):
            fn()
        ev[1].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / reps

    out = {"rows": {"push": nL, "pull": nH}, "f": f, "plain": {}, "bits": {}}
    table = m.tables[1]
    out["plain"]["push_ms"] = timed(lambda: gnn.halo_push(m.graph, H[:nL], lid, table))
    out["plain"]["pull_ms"] = timed(lambda: gnn.halo_pull(m.graph, table, hid, H))
    out["plain"]["bytes_per_row"] = f * es
    for b in (1, 2, 4, 8):
        ldc = gnn.codec_row_bytes(f, b)
        codes = torch.zeros((nT, ldc), dtype=torch.uint8, device="cuda")
        sz = torch.zeros((nT, 2), dtype=torch.float32, device="cuda")
        push_ms = timed(lambda: gnn.halo_push_quantized(m.graph, H[:nL], lid, codes, sz, b, 1234))
        pull_ms = timed(lambda: gnn.halo_pull_quantized(m.graph, codes, sz, b, hid, H))
        row = (f * b + 7) // 8 + 8  # codes + scale / zero point
        push_bytes = nL * (8 + f * es + row)
        pull_bytes = nH * (8 + row + f * es)
        out["bits"][str(b)] = {"push_ms": push_ms, "pull_ms": pull_ms, "bytes_per_row": row,
                               "push_gbs": push_bytes / push_ms / 1e6, "pull_gbs": pull_bytes / pull_ms / 1e6}
        del codes, sz
    m.check_errors()
    return out



def l2_flush_buffer(part, w):
    """A 512 MiB buffer to overwrite between steps when the workload's data could stay in L2 (129 MB), else None."""
    import torch

    es = 2 if w.dtype == "bf16" else 4
    data = 8 * part.nnz + 3 * part.n_total * max(w.widths) * es * len(w.widths)
    if data > 8 * (129 << 20):
        return None
    return torch.zeros(128 << 20, dtype=torch.float32, device="cuda")

def measure_other_schedule(m, stream, steps: int) -> float:
    """ms per step with the other pull / push schedule (sequential if the run overlaps, and the other way)."""
    import torch

    was, side = m.overlap, m.side
    m.overlap = not was
    m.side = torch.cuda.Stream() if m.overlap else None
    try:
        m.step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            m.step()
        e1.record(stream)
        torch.cuda.synchronize()
        m.check_errors()
        return e0.elapsed_time(e1) / steps
    finally:
        m.overlap, m.side = was, side


def measure_other_precision(m, stream, steps: int, ef: int):
    """The step with the activation gradients stored in the other dtype (bf16 <-> fp32; bf16 activations)."""
    import torch

    was = m.grad_dtype
    other = torch.bfloat16 if was == torch.float32 else torch.float32
    m.set_grad_dtype(other)
    try:
        m.step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            m.step()
        e1.record(stream)
        torch.cuda.synchronize()
        m.check_errors()
        ms = e0.elapsed_time(e1) / steps
    finally:
        m.set_grad_dtype(was)
    return {"grad_dtype": "bf16" if other == torch.bfloat16 else "f32", "ms_per_step": ms, "value": ef / (ms / 1e3),
            "steps": steps}


def measure_other_order(m, stream, steps: int, ef: int):
    """The step with the backward of GCN layers l > 0 in the other product order: P = A_hat^T dY gathered in
    bf16, dH = P W^T (bf16 activations, fp32 gradients)."""
    import torch

    from sparse_aggregation_dense_gb300 import gnn

    m.set_reorder(True)
    try:
        m.step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gnn.profile_read(m.graph)  # clear
        gnn.profile_enable(m.graph, True)
        e0.record(stream)
        for _ in range(steps):
            m.step()
        e1.record(stream)
        torch.cuda.synchronize()
        gnn.profile_enable(m.graph, False)
        prof = gnn.profile_read(m.graph)
        m.check_errors()
        ms = e0.elapsed_time(e1) / steps
    finally:
        m.set_reorder(False)
    return {"backward": "dH = (A_hat^T dY) W^T on layers l > 0, P in bf16", "ms_per_step": ms,
            "value": ef / (ms / 1e3), "steps": steps,
            "breakdown_ms_per_step": {k: round(v[0] / steps, 3) for k, v in prof.items()}}


def measure_gat(workload: str, steps: int = 5):
    """A 3-layer graph-attention epoch (GatModel) on another workload: ms per step and edge x feature / s
    (the attention-weighted sums counted like the GCN aggregations)."""
    import torch

    from sparse_aggregation_dense_gb300 import GatModel

    w = workload_by_name(workload)
    part = w.make(SEED)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    widths = list(w.widths)
    m = GatModel(part, widths, tdt, "cuda")
    rng = np.random.default_rng(SEED)
    for l in range(m.L):
        m.tables[l] = torch.empty((part.n_table, m.H[l].stride(0)), dtype=tdt, device="cuda")[:, :widths[l]]
        fill_table(m.tables[l], part.n_table, widths[l], w.dtype == "bf16", SEED, 800 + l, "normal")
        m.W[l].copy_(torch.from_numpy(synth.glorot(widths[l], widths[l + 1], SEED, 810 + l)))
        m.a_src[l].copy_(torch.from_numpy((rng.standard_normal(widths[l + 1]) * 0.3).astype(np.float32)))
        m.a_dst[l].copy_(torch.from_numpy((rng.standard_normal(widths[l + 1]) * 0.3).astype(np.float32)))
    m.H[0][:part.n_local] = m.tables[0][torch.from_numpy(part.local_ids).cuda()]
    m.labels.copy_(torch.from_numpy(synth.labels(part.n_local, widths[-1], SEED, ids=part.local_ids)))
    for _ in range(3):
        m.step()
    m.check_errors()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    e0.record(stream)
    for _ in range(steps):
        m.step()
    e1.record(stream)
    torch.cuda.synchronize()
    m.check_errors()
    ms = e0.elapsed_time(e1) / steps
    ef = part.nnz * 2 * sum(widths[1:])  # the attention-weighted sums, forward and backward, at T's width
    return {"workload": w.name, "widths": widths, "dtype": w.dtype, "grad_dtype": "f32", "ms_per_step": ms,
            "value": ef / (ms / 1e3), "unit": UNIT, "steps": steps,
            "note": f"{len(widths) - 1}-layer single-head GAT epoch (pull, attention forward, push, loss, attention "
                    "backward with halo gradients) through the C ABI"}


def measure_h2d(x_pin, dst, stream, reps: int = 3) -> float:
    """GB/s of the e2e leg's feature copy alone (pinned host -> device)."""
    import torch

    dst.copy_(x_pin, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        dst.copy_(x_pin, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    return x_pin.numel() * x_pin.element_size() * reps / (e0.elapsed_time(e1) / 1e3) / 1e9


def run_ours(args, rank, world, local_rank):
    import torch

    from sparse_aggregation_dense_gb300 import PartitionModel, gnn

    torch.cuda.set_device(local_rank)
    dist = init_dist(world, True)
    w = workload_by_name(args.workload)
    bf = w.dtype == "bf16"
    tdt = torch.bfloat16 if bf else torch.float32
    t_gen = time.time()
    part = w.make(SEED + rank)
    t_gen = time.time() - t_gen
    t_create = time.time()
    gdt = torch.bfloat16 if (bf and args.grad_dtype == "bf16") else torch.float32
    m = PartitionModel(part, w.widths, w.agg, tdt, "cuda", overlap=not args.sequential, narrow=args.narrow,
                       grad_dtype=gdt)
    torch.cuda.synchronize()
    t_create = time.time() - t_create
    for l in range(w.layers):
        stream = synth.STREAM_FEATURES if l == 0 else synth.STREAM_TABLE + l
        m.tables[l] = torch.empty((part.n_table, m.H[l].stride(0)), dtype=tdt, device="cuda")[:, :w.widths[l]]
        fill_table(m.tables[l], part.n_table, w.widths[l], bf, SEED, stream, w.feat_dist if l == 0 else "normal")
    lid = torch.from_numpy(part.local_ids).cuda()
    m.H[0][:part.n_local] = m.tables[0][lid]
    for l in range(w.layers):
        K = (2 if w.agg == "sage" else 1) * w.widths[l]
        m.W[l].copy_(torch.from_numpy(synth.glorot(K, w.widths[l + 1], SEED, synth.STREAM_WEIGHT + l)))
    y = synth.labels(part.n_local, w.widths[-1], SEED, ids=part.local_ids)
    m.labels.copy_(torch.from_numpy(y))
    torch.cuda.synchronize()

    ef = edge_feat_per_step(part, w)
    for _ in range(args.warmup):
        m.step()
    m.check_errors()
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gnn.profile_read(m.graph)  # clear
    gnn.profile_enable(m.graph, True)
    launches0 = gnn.launch_count()
    barrier(dist, True)
    torch.cuda.synchronize()
    flush = l2_flush_buffer(part, w)
    with ClockSampler(torch.cuda.current_device()) as clk:
        if flush is None:
            ev0.record(stream)
            for _ in range(args.steps):
                m.step()
            ev1.record(stream)
            torch.cuda.synchronize()
            ms_total = ev0.elapsed_time(ev1)
        else:  # L2-sized workload: flush L2 before every step, time the steps only
            ms_total = 0.0
            for _ in range(args.steps):
                flush.add_(1)
                ev0.record(stream)
                m.step()
                ev1.record(stream)
                torch.cuda.synchronize()
                ms_total += ev0.elapsed_time(ev1)
    barrier(dist, True)
    launches = gnn.launch_count() - launches0
    gnn.profile_enable(m.graph, False)
    prof = gnn.profile_read(m.graph)
    m.check_errors()
    ms_local = ms_total / args.steps
    ms = max_over_ranks(dist, ms_local, True)
    total_ef = sum_over_ranks(dist, float(ef), True)
    value = total_ef / (ms / 1e3)

    # dominant kernel: the aggregation (forward + backward launches)
    hbm, bf16_tf, peak_kind = measured_peaks()
    fwd_b, bwd_b = aggregation_bytes(part, w, 2 if bf else 4, args.narrow, 2 if gdt == torch.bfloat16 else 4)
    alg_bytes = (sum(fwd_b) + sum(bwd_b)) * args.steps
    agg_ms = prof["agg_fwd"][0] + prof["agg_bwd"][0]
    agg_launches = prof["agg_fwd"][1] + prof["agg_bwd"][1]
    achieved = alg_bytes / (agg_ms / 1e3) / 1e9 if agg_ms > 0 else 0.0
    traffic = ncu_traffic(w.name, "bf16" if gdt == torch.bfloat16 else "f32")
    l2 = int(getattr(torch.cuda.get_device_properties(torch.cuda.current_device()), "L2_cache_size", 0) or 0)
    cache_aware = None
    if l2 > 0 and agg_ms > 0:
        floor_b = sum(cache_floor_bytes(part, w, 2 if bf else 4, 2 if gdt == torch.bfloat16 else 4, l2, args.narrow))
        ach = floor_b / (agg_ms / args.steps / 1e3) / 1e9
        cache_aware = {"model": "ideal static cache of the L2 size holding the most-gathered rows, every other "
                                "gather from DRAM, streamed terms once", "l2_bytes": l2, "bytes_per_step": floor_b,
                       "achieved": ach, "frac": ach / hbm if hbm else None}
    breakdown = {k: round(v[0] / args.steps, 3) for k, v in prof.items()}
    breakdown["other"] = round(ms_local - sum(v[0] for v in prof.values()) / args.steps, 3)

    # end to end through the C ABI from pinned host buffers
    nL = part.n_local
    ld0 = m.H[0].stride(0)
    x_host = synth.features(0, w.widths[0], ld0, SEED, synth.STREAM_FEATURES, w.feat_dist, bf16=bf,
                            ids=part.local_ids)
    x_pin = torch.from_numpy(x_host.view(np.int16) if bf else x_host).pin_memory()
    if bf:
        x_pin = x_pin.view(torch.bfloat16)
    y_pin = torch.from_numpy(y).pin_memory()
    loss_pin = torch.empty(1, dtype=torch.float32).pin_memory()
    dw_pin = [torch.empty(d.shape, dtype=torch.float32).pin_memory() for d in m.dW]
    h0 = m.H[0].as_strided((part.n_total, ld0), (ld0, 1))[:nL]
    e2e_steps = max(1, args.steps)  # as many steps as the device-timed leg
    barrier(dist, True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    # the first step's inputs are copied before it; every later step's inputs are staged during the step
    # before it (features once layer 0 has read them, labels once the loss has), on a copy stream
    h0.copy_(x_pin, non_blocking=True)
    m.labels.copy_(y_pin, non_blocking=True)
    for i in range(e2e_steps):
        if i + 1 < e2e_steps:
            m.stage_inputs(x_pin, y_pin)
        m.step()
        loss_pin.copy_(m.loss, non_blocking=True)
        for d, hp in zip(m.dW, dw_pin):
            hp.copy_(d, non_blocking=True)
        stream.synchronize()  # the host reads the step's result
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1) / e2e_steps, True)
    if args.quick:  # tuning runs: the timed step and its breakdown only
        codec, other_ms, other_prec, other_order, h2d_gbs = None, float("nan"), None, None, float("nan")
    else:
        codec = measure_codec(m, part, w, tdt, stream)
        other_ms = measure_other_schedule(m, stream, max(3, min(args.steps, 5)))
        other_prec = measure_other_precision(m, stream, max(3, min(args.steps, 5)), ef) if bf and not args.narrow \
            else None
        other_order = measure_other_order(m, stream, max(3, min(args.steps, 5)), ef) \
            if bf and w.agg == "gcn" and gdt == torch.float32 and not args.narrow else None
        h2d_gbs = measure_h2d(x_pin, h0, stream)
    gat = None if (args.quick or not args.gat_workload) else \
        [measure_gat(x) for x in args.gat_workload.split(",") if x]
    h2d = int(x_pin.numel() * x_pin.element_size() + y_pin.numel() * 4)
    d2h = int(4 + sum(d.numel() * 4 for d in m.dW))

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_entry(part, w, args.cpu_seconds)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded generators, shapes of the pages' workloads)",
        "config": {
            "workload": w.name,
            "description": w.description,
            "n_local": part.n_local, "n_halo": part.n_halo, "nnz": part.nnz, "n_table": part.n_table,
            "widths": w.widths, "agg": w.agg,
            "edge_feat_per_step": ef,
            "parallelism": f"one partition per GPU x{world} (no data-path collective)",
            "l2": ("inputs larger than L2 (no flush)" if flush is None
                   else "L2 flushed before every timed step (512 MiB written); steps timed one by one"),
            "seed": SEED,
            "layer_order": "multiplication first on narrowing GCN layers" if args.narrow else "aggregation first",
            "grad_dtype": "bf16" if gdt == torch.bfloat16 else "f32",
            "precision": ("bf16 activations (features, tables, Z, layer outputs), "
                          + ("bf16" if gdt == torch.bfloat16 else "fp32") + " activation gradients (G, dZ, dH), "
                          "fp32 accumulation, fp32 dW") if bf else "fp32 throughout",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "aggregation (CSR SpMM + heavy-row fix-up), forward and backward launches",
            "achieved": achieved,
            "peak": hbm,
            "unit": "GB/s",
            "frac": achieved / hbm if hbm else None,
            "traffic": traffic,
            "traffic_scope": "DRAM bytes of one step's aggregation launches (ncu summary in profiles/)",
            "dram_achieved": (traffic / (agg_ms / args.steps / 1e3) / 1e9) if (traffic and agg_ms > 0) else None,
            "dram_frac": (traffic / (agg_ms / args.steps / 1e3) / 1e9 / hbm) if (traffic and agg_ms > 0 and hbm)
            else None,
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)",
            "algorithmic_bytes_per_step": sum(fwd_b) + sum(bwd_b),
            "launch_groups": agg_launches,
            "ms_per_step": round(agg_ms / args.steps, 3),
            "cache_aware": cache_aware,
            "traffic_small_case": small_case_traffic(),
        },
        "breakdown_ms_per_step": breakdown,
        "breakdown_note": "library event timing per kernel group; in the overlapped schedule pull and push run "
                          "beside the layers, so the groups can sum to more than the step ('other' < 0)",
        "cpu_baseline": cpu,
        "e2e": {"value": total_ef / (e2e_ms / 1e3), "unit": UNIT, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "input_staging": "each step's inputs after the first are copied during the step before it, on a "
                                 "copy stream (features once layer 0 has read H[0], labels once the loss has)",
                "h2d_gbs_feature_copy_alone": round(h2d_gbs, 1)},
        "other_precision": other_prec,
        "other_order": other_order,
        "gat": gat,
        "gpu_launches": int(launches),
        "halo_codec": codec,
        "schedule": "sequential" if args.sequential else "overlapped (pulls and pushes on a second stream)",
        "other_schedule": {"schedule": "overlapped" if args.sequential else "sequential", "ms_per_step": other_ms,
                           "value": total_ef / (other_ms / 1e3), "note": "same results as the timed step"},
        "clocks": clk.summary(),
        "setup_s": {"generate": round(t_gen, 1), "graph_create_and_alloc": round(t_create, 1)},
    }
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle

    w = workload_by_name(args.workload)
    part = w.make(SEED)
    ef_total, secs = 0, 0.0
    desc = ""
    for i in range(args.warmup + args.steps):
        ef, s, desc = oracle_sample(part, w, args.ref_seconds, SEED + 7 * i, max_batches=16)
        if i >= args.warmup:
            ef_total += ef
            secs += s
    value = ef_total / secs
    ms_full = edge_feat_per_step(part, w) / value * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_full, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded generators, shapes of the pages' workloads)",
        "config": {"workload": w.name, "description": w.description, "n_local": part.n_local,
                   "n_halo": part.n_halo, "nnz": part.nnz, "widths": w.widths, "agg": w.agg,
                   "note": "ms_per_step extrapolated per edge from the sampled rows"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def gather_ceiling(reps: int = 5):
    """Throughput of the aggregation kernel on uniform random columns (2^21 rows of 48 entries) gathered from
    tables of 2^15 .. 2^23 rows: from tables that L2 holds the kernel's own per-entry limit, from tables far
    larger than L2 its DRAM-bound rate.  Prints one JSON line."""
    import numpy as np
    import torch
    from sparse_aggregation_dense_gb300 import gnn, padded

    torch.cuda.set_device(0)
    nL, deg = 1 << 21, 48
    rng = np.random.default_rng(SEED)
    rows = []
    for K in (1 << 15, 1 << 18, 1 << 21, 1 << 23):
        cols = np.sort(rng.integers(0, K, (nL, deg), dtype=np.int64), axis=1).astype(np.int32).ravel()
        rowptr = (np.arange(nL + 1, dtype=np.int64) * deg).astype(np.int32)
        nH = max(0, K - nL)  # every column id is below n_local + n_halo
        g = gnn.graph_create(torch.from_numpy(rowptr).cuda(), torch.from_numpy(cols).cuda(), nL, nH, None, "gcn")
        for f, dt in ((128, torch.bfloat16), (256, torch.bfloat16), (256, torch.float32)):
            H = padded(nL + nH, f, dt, "cuda")
            H.normal_()
            Z = padded(nL, f, dt, "cuda")
            for _ in range(3):
                gnn.aggregate_forward_noalloc(g, H, Z)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                gnn.aggregate_forward_noalloc(g, H, Z)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            rb = f * (2 if dt == torch.bfloat16 else 4)
            rows.append({"table_rows": K, "table_mb": round(K * rb / 2**20), "row_bytes": rb, "ms": round(ms, 3),
                         "entries_per_s": nL * deg / (ms / 1e3), "gathered_tbs": nL * deg * rb / (ms / 1e3) / 1e12})
            del H, Z
        if gnn.get_error(g) != gnn.GNN_OK:
            raise RuntimeError("device error word set")
        gnn.graph_destroy(g)
        torch.cuda.empty_cache()
    print(json.dumps({"gather_ceiling": rows, "entries": nL * deg,
                      "note": "aggregation kernel (gnn_aggregate_forward_noalloc), uniform random columns"}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="rmat16m")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle work timed for cpu_baseline")
    ap.add_argument("--ref-seconds", type=float, default=3.0, help="oracle work per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--gat-workload", default="rmat131k,sage2m",
                    help="workloads (comma-separated) of the graph-attention epochs reported beside the step "
                         "('' to skip)")
    ap.add_argument("--quick", action="store_true",
                    help="time the step only (no codec, other schedule, other precision or H2D figures)")
    ap.add_argument("--narrow", action="store_true",
                    help="GCN layers whose output is narrower than their input multiply first: A (H W)")
    ap.add_argument("--grad-dtype", choices=["f32", "bf16"], default="f32",
                    help="storage of the activation gradients of bf16 workloads (default fp32)")
    ap.add_argument("--sequential", action="store_true",
                    help="pulls and pushes in line on the compute stream instead of on a second stream")
    ap.add_argument("--gather-ceiling", action="store_true",
                    help="measure the aggregation's gather throughput on uniform random columns and exit")
    ap.add_argument("--gat-only", action="store_true",
                    help="time the graph-attention epoch of --gat-workload alone and exit")
    args = ap.parse_args(argv)
    if args.gather_ceiling:
        return gather_ceiling()
    if args.gat_only:
        import torch

        torch.cuda.set_device(0)
        print(json.dumps({"gat": [measure_gat(x, steps=max(1, args.steps)) for x in args.gat_workload.split(",")
                                  if x]}))
        return None
    if args.narrow and args.grad_dtype != "bf16" and workload_by_name(args.workload).dtype == "bf16":
        args.grad_dtype = "bf16"  # the multiplication-first layers keep their gradients in the activations' dtype
    if args.warmup < 3 and args.impl == "ours" and not args.workload.endswith("-tiny"):
        args.warmup = 3
    rank, world, local_rank = rank_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
