"""Helpers shared by the GPU parity tests: inputs from the generators, the same
inputs widened for the oracle, and the elementwise tolerance check."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from sparse_aggregation_dense_gb300 import gnn, ld_for

TOL = {"f32": 1e-4, "bf16": 2e-2}


def close(gpu: np.ndarray, ref: np.ndarray, tol: float, what: str = ""):
    """|x - r| <= tol * (|r| + rms(r)) elementwise (rms over the compared values)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if ref.size == 0:
        return
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(gpu - ref)
    bound = tol * (np.abs(ref) + rms)
    bad = err > bound
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"gpu {gpu[tuple(i)]!r} ref {ref[tuple(i)]!r} (rms {rms:.3g})")


def close_mostly(gpu: np.ndarray, ref: np.ndarray, tol: float, what: str = "", max_frac: float = 0.01,
                 norm_tol: float = 1e-2):
    """For chained bf16 results, where a ReLU mask decision may flip between the
    two sides (pre-activations within a bf16 rounding of zero): at most max_frac of
    the elements may fall outside the elementwise bound, and the relative
    Frobenius error must stay within norm_tol."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if ref.size == 0:
        return
    rms = float(np.sqrt(np.mean(ref * ref)))
    bad = np.abs(gpu - ref) > tol * (np.abs(ref) + rms)
    frac = float(bad.mean())
    nrm = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300))
    assert frac <= max_frac and nrm <= norm_tol, f"{what}: {frac:.4%} outside, relative norm error {nrm:.3g}"


def torch_dtype(dt: str):
    return torch.bfloat16 if dt == "bf16" else torch.float32


def gen_matrix(rows: int, f: int, dt: str, seed: int, stream: int, dist: str = "normal", ids=None):
    """Host matrix (rows x ld) in storage form (uint16 bf16 bits or float32)."""
    ld = ld_for(f, torch_dtype(dt))
    return synth.features(rows, f, ld, seed, stream, dist, bf16=(dt == "bf16"), ids=ids)


def to_device(host: np.ndarray, dt: str, f: int) -> torch.Tensor:
    """Device copy of a generator matrix, returned as its (rows x f) view."""
    if dt == "bf16":
        t = torch.from_numpy(host.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        t = torch.from_numpy(host).cuda()
    return t[:, :f]


def to_host(t: torch.Tensor) -> np.ndarray:
    """float64 host copy of a device view."""
    return t.float().cpu().numpy().astype(np.float64)


def widen(host: np.ndarray, dt: str, f: int) -> np.ndarray:
    return oracle.widen(host[:, :f], dt == "bf16")


def maybe_round(x: np.ndarray, dt: str) -> np.ndarray:
    return oracle.round_bf16(x) if dt == "bf16" else x


def sample_with_heavy(rowptr: np.ndarray, k: int, seed: int, extra_top: int = 8) -> np.ndarray:
    """k random rows plus the heaviest rows and rows just above the split threshold."""
    n = rowptr.shape[0] - 1
    rows = set(synth.sample_rows(n, k, seed).tolist())
    deg = np.diff(rowptr)
    order = np.argsort(-deg, kind="stable")
    rows.update(order[:extra_top].tolist())
    for lo, hi in ((512, 520), (1024, 1100), (2048, 4096)):
        cand = np.nonzero((deg > lo) & (deg <= hi))[0]
        rows.update(cand[:4].tolist())
    rows.update([0, n - 1] if n else [])
    return np.array(sorted(rows), dtype=np.int64)


def column_subset(rowptr: np.ndarray, colidx: np.ndarray, rows: np.ndarray, n_cols: int):
    """Columns used by `rows` and a map column -> position (for oracle hmap)."""
    if rows.size == 0:
        return np.zeros(0, np.int64), -np.ones(n_cols, np.int64)
    parts = [colidx[rowptr[r]:rowptr[r + 1]] for r in rows]
    cols = np.unique(np.concatenate(parts).astype(np.int64)) if parts else np.zeros(0, np.int64)
    cmap = -np.ones(n_cols, np.int64)
    cmap[cols] = np.arange(cols.shape[0])
    return cols, cmap


def assert_ok(g) -> None:
    """The graph's device error status is clean; on a CUDA failure, say which."""
    st = gnn.get_error(g)
    assert st == gnn.GNN_OK, f"status {st}: {gnn.last_cuda_error() if st == gnn.GNN_ECUDA else 'device error word set'}"
